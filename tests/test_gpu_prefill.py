"""GPU parity of the prefill path (block-scaled FP4 x FP4 tensor-core GEMMs) against the oracle.

Prefill quantises x and the SwiGLU output h to NVFP4 (16-element E4M3 block
scales, tensor scale 1).  x is quantised from exact bf16 values with the same
fp32 operations on both sides, so its codes must agree exactly (checked
through the outputs).  h is computed in fp32 by the tensor cores and in fp64
by the oracle; where the oracle's scaled value sits within a hair of an E2M1
rounding midpoint the GPU may legitimately round the other way.  The check is
therefore two-stage:

  1. every h code the GPU produced equals the oracle's, except at elements the
     oracle itself flags as near a midpoint, where it must equal the oracle's
     alternative (the other neighbour); block scales must match exactly;
  2. y must match the oracle's y recomputed with those oracle-determined
     alternatives, within the decode tolerances.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import moe as omoe
from oracle import nvfp4 as onv
from tests import harness

pytestmark = pytest.mark.gpu

SMALL = synth.MoEShape(d_model=256, n_experts=16, top_k=2, d_ff=256, n_shared=1)
F32 = np.float32
MID_TOL = 2e-4    # relative distance to an E2M1 rounding midpoint treated as a near-tie


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import nvfp4_expert_ffn_gemv_b300 as lib
    return lib


def _oracle_h(lw, e, x_row):
    """fp32 h of expert e for one token (x quantised), plus its oracle NVFP4 codes/scales."""
    wg, wu, _ = lw.expert(int(e))
    h = omoe.expert_hidden(wg, wu, x_row[None, :], quant_act=True)[0].astype(F32)
    codes, scales = onv.quantize_activation(h[None, :])
    return h, onv.unpack_codes(codes)[0], scales[0]


def _block_codes(hb, scale_code):
    """Oracle codes of one 16-element block under a given E4M3 scale, and per element the
    alternative code when the scaled value lies within MID_TOL of an E2M1 midpoint (else -1)."""
    d = F32(onv.e4m3_decode(np.array([scale_code]))[0])
    if d == 0:
        return np.zeros(16, np.int64), np.full(16, -1, np.int64)
    v = (hb.astype(F32) / d).astype(F32)
    codes = onv.e2m1_encode(v).astype(np.int64)
    alt = np.full(16, -1, np.int64)
    grid = onv.E2M1_TABLE[:8]
    mag = np.abs(v.astype(np.float64))
    chosen = codes & 7
    for lo in range(7):
        mid = (grid[lo] + grid[lo + 1]) / 2
        near = np.abs(mag - mid) <= MID_TOL * mid
        other = np.where(chosen == lo, lo + 1, lo)
        sign = np.where((v < 0) & (other != 0), 8, 0)
        alt = np.where(near, other | sign, alt)
    return codes, alt


def _scale_alternative(hb):
    """The other E4M3 neighbour when amax/6 lies within MID_TOL of an E4M3 midpoint, else None."""
    q = F32(np.max(np.abs(hb.astype(F32))) / F32(6.0))
    code = int(onv.e4m3_encode(np.array([q]))[0])
    grid = onv.E4M3_TABLE[:0x7F]
    for lo in (code - 1, code):
        if 0 <= lo < len(grid) - 1:
            mid = (grid[lo] + grid[lo + 1]) / 2
            if abs(float(q) - mid) <= MID_TOL * mid:
                return lo + 1 if lo == code else lo
    return None


def _match_h(h32, gpu_codes, gpu_scales, t):
    """Stage 1 for one slot: every GPU block scale and code must be the oracle's or the oracle's
    own near-tie alternative.  Returns the codes and scales the oracle accepts (fp64 dequantised h)
    and the number of elements that took the alternative."""
    f = h32.shape[0]
    codes = np.zeros(f, np.int64)
    flips = 0
    for b in range(f // 16):
        hb = h32[16 * b:16 * b + 16]
        sc_o = int(onv.quantize_activation(hb[None, :])[1][0, 0])
        sc = int(gpu_scales[b])
        if sc != sc_o:
            assert _scale_alternative(hb) == sc, f"token {t}: block scale {sc} is not a near-tie of {sc_o}"
        cb, alt = _block_codes(hb, sc)
        g = gpu_codes[16 * b:16 * b + 16].astype(np.int64)
        diff = np.nonzero(g != cb)[0]
        assert np.all(alt[diff] >= 0), f"token {t}: h codes differ away from a rounding midpoint"
        assert np.array_equal(g[diff], alt[diff]), f"token {t}: unexpected h code"
        cb[diff] = alt[diff]
        codes[16 * b:16 * b + 16] = cb
        flips += len(diff) + (sc != sc_o) * 16
    hq = onv.dequantize(onv.pack_codes(codes[None, :].astype(np.uint8)), gpu_scales[None, :], 1.0)[0]
    return hq, flips


def _check_prefill(lib, layer, xb, x, T, sample=None):
    s = layer.shape
    k, S, f = s.top_k, s.n_shared, s.d_ff
    y = torch.empty((T, s.d_model), dtype=torch.bfloat16, device="cuda")
    lib.moe_forward_prefill(layer.ctx, xb, T, y)
    slots = T * (k + S)
    hc = torch.empty((slots, f // 2), dtype=torch.uint8, device="cuda")
    hs = torch.empty((slots, f // 16), dtype=torch.uint8, device="cuda")
    lib.moe_debug_prefill_h(layer.ctx, T, hc, hs)
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    wsel = torch.empty((T, k), dtype=torch.float32, device="cuda")
    lib.moe_debug_routing(layer.ctx, T, idx, wsel)     # the experts this prefill used
    torch.cuda.synchronize()
    assert lib.moe_get_device_status(layer.ctx) == 0
    idx = idx.cpu().numpy()
    hc = onv.unpack_codes(hc.cpu().numpy())
    hs = hs.cpu().numpy()
    y = y.float().cpu().numpy()
    tokens = range(T) if sample is None else sample
    used = set(idx[list(tokens)].ravel().tolist()) | set(range(s.n_experts, s.n_all))
    lw = layer.oracle_weights(sorted(used))
    flips = 0
    y_ref, y_gpu = [], []
    for t in tokens:
        xt = x[t]
        r = omoe.moe_layer(lw, xt[None, :], k, S, prefill=True)
        assert np.array_equal(r.idx[0], idx[t]) or r.near_tie[0], f"routing of token {t}"
        slot_list = [(t * k + j, int(idx[t, j]), float(r.w[0, j])) for j in range(k)]
        slot_list += [(T * k + i * T + t, s.n_experts + i, 1.0) for i in range(S)]
        yt = np.zeros(s.d_model)
        for slot, e, wj in slot_list:
            h32, _, _ = _oracle_h(lw, e, xt)
            hq, nf = _match_h(h32, hc[slot], hs[slot], t)
            flips += nf
            _, _, wd = lw.expert(e)
            yt += wj * (np.asarray(wd, np.float64) @ hq)
        y_ref.append(onv.bf16_rne(yt))
        y_gpu.append(y[t])
    rel, mx = harness.compare(torch.tensor(np.array(y_gpu)), np.array(y_ref))
    assert rel <= harness.REL_L2_TOL and mx <= harness.MAX_ABS_RMS_TOL, f"rel_l2={rel:.3e} max_abs/rms={mx:.3e}"
    return rel, mx, flips


@pytest.mark.parametrize("T", [1, 37, 300])
def test_prefill_small(lib, T):
    layer = harness.make_layer(lib, SMALL, seed=11, router_seed=12, fmt=0, max_tokens=512)
    try:
        xb, x = synth.tokens(SMALL, T, seed=200 + T)
        _check_prefill(lib, layer, xb.cuda(), x.double().numpy(), T)
    finally:
        lib.moe_destroy(layer.ctx)


@pytest.mark.parametrize("T", [1024, 1500])
def test_bucketing_grid_path(lib, T):
    """From 1024 tokens the bucketing runs as three grids (count, scan, scatter):
    the per-expert counts equal the histogram of the chosen experts, and the
    prefill output, which reads every position the scatter wrote, matches the
    oracle on sampled tokens (T = 1500 leaves a ragged last chunk)."""
    layer = harness.make_layer(lib, SMALL, seed=21, router_seed=22, fmt=0, max_tokens=2048)
    try:
        k, E = SMALL.top_k, SMALL.n_experts
        xb, x = synth.tokens(SMALL, T, seed=400 + T)
        idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
        w = torch.empty((T, k), dtype=torch.float32, device="cuda")
        counts = torch.empty((E,), dtype=torch.int32, device="cuda")
        lib.moe_route(layer.ctx, xb.cuda(), T, idx, w, counts)
        torch.cuda.synchronize()
        assert lib.moe_get_device_status(layer.ctx) == 0
        hist = np.bincount(idx.cpu().numpy().ravel(), minlength=E)
        assert np.array_equal(counts.cpu().numpy(), hist)
        sample = [0, 1, T // 2, T - 1] + list(range(5, T, 97))
        _check_prefill(lib, layer, xb.cuda(), x.double().numpy(), T, sample=sample)
    finally:
        lib.moe_destroy(layer.ctx)


def test_prefill_flint_4096_sampled(lib):
    s = synth.FLINT
    layer = harness.make_layer(lib, s, seed=synth.layer_seed(0), router_seed=synth.router_seed(0), fmt=0,
                               max_tokens=4096)
    try:
        xb, x = synth.tokens(s, 4096, seed=synth.token_seed(7))
        sample = [0, 1, 777, 2048, 4095] + list(range(100, 4096, 1013))
        rel, mx, flips = _check_prefill(lib, layer, xb.cuda(), x.double().numpy(), 4096, sample=sample)
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
