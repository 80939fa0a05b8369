"""Pins of the oracle's MoE layer against brute force, closed forms and invariants.

* top-k: exhaustive search over all C(E, k) subsets on tiny E, with integer
  logits that force exact ties (the chosen set is the max-sum subset that is
  lexicographically smallest; the order is by descending logit, ties to the
  lower index);
* combine weights: equal to the full softmax over all experts renormalised
  over the chosen ones (scipy's softmax), summing to one;
* bucketing: against np.bincount and a direct sort;
* experts: a one-hot router reproduces one dense SwiGLU computed with plain
  Python loops and math.fsum (exactly rounded sums); k = E with equal logits
  gives the mean of the experts; identical experts give expert + shared;
* silu against scipy's expit; the prefill path equals the decode path when
  x and h are already representable in NVFP4 with unit tensor scale.
"""
import itertools
import math

import numpy as np
import pytest
import scipy.special

from oracle import moe, nvfp4

F32 = np.float32


def test_top_k_brute_force_with_ties():
    rng = np.random.default_rng(5)
    for E, k in ((16, 2), (8, 3), (6, 6), (5, 1)):
        for _ in range(60):
            logits = rng.integers(-3, 4, size=(1, E)).astype(F32)   # many exact ties
            idx = moe.top_k(logits, k)[0]
            best = None
            for sub in itertools.combinations(range(E), k):
                key = (-sum(float(logits[0, e]) for e in sub), sub)
                if best is None or key < best:
                    best = key
            assert tuple(sorted(idx.tolist())) == best[1]
            vals = logits[0, idx]
            assert np.all(np.diff(vals) <= 0)
            for a in range(k - 1):
                if vals[a] == vals[a + 1]:
                    assert idx[a] < idx[a + 1]


def test_combine_weights_equal_renormalised_full_softmax():
    rng = np.random.default_rng(6)
    logits = (rng.standard_normal((40, 256)) * 0.9).astype(F32)
    idx = moe.top_k(logits, 6)
    w = moe.combine_weights(logits, idx)
    full = scipy.special.softmax(logits.astype(np.float64), axis=1)
    sel = np.take_along_axis(full, idx.astype(np.int64), axis=1)
    ref = sel / sel.sum(axis=1, keepdims=True)
    assert np.allclose(w, ref, rtol=1e-13, atol=0)
    assert np.all(np.abs(w.sum(axis=1) - 1) < 6 * 2.0 ** -52 * 4)
    assert np.all(np.diff(w, axis=1) <= 0)


def test_bucket_against_bincount_and_sort():
    rng = np.random.default_rng(7)
    T, k, E = 37, 6, 64
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    counts, offsets, perm = moe.bucket(idx, E)
    assert np.array_equal(counts, np.bincount(idx.ravel(), minlength=E))
    assert offsets[0] == 0 and offsets[-1] == T * k and np.array_equal(np.diff(offsets), counts)
    flat = idx.ravel()
    ref = sorted(range(T * k), key=lambda s: (flat[s], s))
    assert perm.tolist() == ref


def _dense_swiglu_loops(wg, wu, wd, x):
    """Textbook SwiGLU with explicit loops and exactly rounded sums."""
    f, d = len(wg), len(x)
    h = []
    for j in range(f):
        g = math.fsum(wg[j][i] * x[i] for i in range(d))
        u = math.fsum(wu[j][i] * x[i] for i in range(d))
        h.append(g / (1.0 + math.exp(-g)) * u)
    return [math.fsum(wd[r][j] * h[j] for j in range(f)) for r in range(len(wd))]


def _tiny_layer(rng, d=32, f=16, E=8, shared=1, bias=None):
    n = E + shared
    wg = (rng.standard_normal((n, f, d)) * 0.2).astype(F32)
    wu = (rng.standard_normal((n, f, d)) * 0.2).astype(F32)
    wd = (rng.standard_normal((n, d, f)) * 0.2).astype(F32)
    router = (rng.standard_normal((d, E)) * 0.2).astype(F32)
    return moe.quantize_layer(wg, wu, wd, router, bias)


def test_one_hot_router_reproduces_dense_expert():
    rng = np.random.default_rng(8)
    E, target = 8, 5
    bias = np.full(E, -1e4, F32)
    bias[target] = 1e4
    lw = _tiny_layer(rng, E=E, shared=0, bias=bias)
    x = nvfp4.bf16_rne(rng.standard_normal((3, 32)))
    r = moe.moe_layer(lw, x, k=1, n_shared=0)
    assert np.all(r.idx[:, 0] == target) and np.all(r.w == 1.0)
    wg, wu, wd = (m.tolist() for m in lw.expert(target))
    for t in range(3):
        ref = _dense_swiglu_loops(wg, wu, wd, x[t].tolist())
        assert np.allclose(r.y[t], ref, rtol=1e-12, atol=1e-15)


def test_k_equals_e_with_equal_logits_gives_mean_plus_shared():
    rng = np.random.default_rng(9)
    E = 6
    lw = _tiny_layer(rng, E=E, shared=1)
    lw.router[:] = 0
    x = nvfp4.bf16_rne(rng.standard_normal((2, 32)))
    r = moe.moe_layer(lw, x, k=E, n_shared=1)
    assert np.allclose(r.w, 1.0 / E, rtol=1e-15)
    ref = sum(moe.swiglu_expert(*lw.expert(e), x) for e in range(E)) / E
    ref = ref + moe.swiglu_expert(*lw.expert(E), x)
    assert np.allclose(r.y, ref, rtol=1e-12, atol=1e-15)


def test_identical_experts_give_expert_plus_shared():
    rng = np.random.default_rng(10)
    lw = _tiny_layer(rng, E=8, shared=1)
    for t in (lw.gate, lw.up, lw.down):
        t.codes[:8] = t.codes[0]
        t.scales[:8] = t.scales[0]
        t.ts[:8] = t.ts[0]
    x = nvfp4.bf16_rne(rng.standard_normal((4, 32)))
    r = moe.moe_layer(lw, x, k=3, n_shared=1)
    ref = moe.swiglu_expert(*lw.expert(0), x) + moe.swiglu_expert(*lw.expert(8), x)
    assert np.allclose(r.y, ref, rtol=1e-12, atol=1e-15)


def test_silu():
    z = np.linspace(-30, 30, 1001)
    assert np.allclose(moe.silu(z), z * scipy.special.expit(z), rtol=1e-14, atol=1e-300)
    assert moe.silu(0.0) == 0.0
    assert moe.silu(-800.0) == 0.0 and moe.silu(800.0) == 800.0


def test_prefill_quantises_x_and_h_closed_form():
    # x = [6, 3, 1.5, 0.5, 0...] is exact in NVFP4 (block amax 6 -> scale 1).
    # W_gate = 64 I, W_up = I, W_down = I: g = 64 x, u = x, h = silu(64 x) x
    # ~= [2304, 576, 144, 16].  h's block amax 2304 gives the E4M3 scale
    # 2304 / 6 = 384 exactly, h / 384 ~= [6, 1.5, 0.375, 0.042] rounds to
    # [6, 1.5, 0.5, 0] on the E2M1 grid, so the prefill output is exactly
    # [2304, 576, 192, 0, ...] while decode keeps h unquantised.
    d = 16
    x = np.zeros((1, d))
    x[0, :4] = [6.0, 3.0, 1.5, 0.5]
    eye = np.eye(d)
    y_pre = moe.swiglu_expert(eye * 64.0, eye, eye, x, quant_act=True)
    assert y_pre[0, :4].tolist() == [2304.0, 576.0, 192.0, 0.0] and not y_pre[0, 4:].any()
    y_dec = moe.swiglu_expert(eye * 64.0, eye, eye, x)
    ref = [v * 64 * v / (1 + math.exp(-64 * v)) for v in (6.0, 3.0, 1.5, 0.5)]
    assert np.allclose(y_dec[0, :4], ref, rtol=1e-15)
    # a non-representable x is quantised first: 0.3 -> block scale 0.05 -> codes of 0.3/0.05 = 6
    x2 = np.zeros((1, d))
    x2[0, 0] = 0.3
    xq_c, xq_s = nvfp4.quantize_activation(x2.astype(F32))
    assert nvfp4.e4m3_decode(xq_s)[0, 0] == nvfp4.E4M3_TABLE[nvfp4.e4m3_encode(np.array([F32(0.3) / F32(6)]))[0]]


def test_near_tie_flag():
    logits = np.array([[3.0, 2.0, 2.0 + 5e-7, 1.0], [3.0, 2.0, 1.0, 0.0]], F32)
    flags = moe.near_ties(logits, 2)
    assert flags.tolist() == [True, False]


def test_stack_residual_is_bf16():
    rng = np.random.default_rng(11)
    layers = [_tiny_layer(rng, E=8, shared=1) for _ in range(3)]
    x = nvfp4.bf16_rne(rng.standard_normal((2, 32)))
    out, res = moe.moe_stack(layers, x, k=2)
    assert np.array_equal(out, nvfp4.bf16_rne(out))
    x1 = moe.residual(x, res[0].y)
    assert np.array_equal(x1, nvfp4.bf16_rne(x + res[0].y))
