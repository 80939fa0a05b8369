"""Pins of both oracles -- the C++ one (oracle/moe_oracle.cpp, the reference the GPU
tests use) and the numpy fp64 one (oracle/moe.py, its cross-check) -- against
things other than themselves:

* router_logits: textbook loops with math.fsum (exactly rounded sums) on tiny
  inputs, with and without a bias; a dropped x.W_r term, a bias added twice, a
  transposed router or a wrong index all fail here;
* the expert's SwiGLU hidden vector h (numpy ``expert_hidden``, C++
  ``or_expert``): textbook fsum loops, with the activation quantiser on and off;
* top-k: exhaustive search over every k-subset on tiny E with integer logits
  (forced exact ties), signed zeros, NaN (ranked below every number);
* combine weights: scipy's softmax over all experts renormalised;
* bucketing: np.bincount and a direct sort;
* the C++ codec: torch's float8_e4m3fn conversions on every code and midpoint,
  a brute-force nearest search over the 16 E2M1 codes, torch's bf16 rounding;
* the C++ layer: a one-hot router reproduces one dense SwiGLU computed with
  fsum loops, k = E with equal logits gives the mean of the experts, identical
  experts give expert + shared, results do not depend on the thread count, and
  the whole layer agrees with the numpy oracle (indices exactly).
"""
import itertools
import math

import numpy as np
import pytest
import scipy.special
import torch

from oracle import cpp, moe, nvfp4

F32 = np.float32


def _fsum_logits(x, router, bias):
    T, d = x.shape
    E = router.shape[1]
    out = np.empty((T, E))
    for t in range(T):
        for e in range(E):
            s = math.fsum(float(x[t, i]) * float(router[i, e]) for i in range(d))
            out[t, e] = s + (float(bias[e]) if bias is not None else 0.0)
    return out


@pytest.mark.parametrize("impl", ["cpp", "numpy"])
@pytest.mark.parametrize("with_bias", [False, True])
def test_router_logits_against_fsum_loops(impl, with_bias):
    rng = np.random.default_rng(31)
    T, d, E = 5, 48, 7
    x = nvfp4.bf16_rne(rng.standard_normal((T, d))).astype(F32)
    router = (rng.standard_normal((d, E)) * 0.3).astype(F32)
    bias = (rng.standard_normal(E) * 2.0).astype(F32) if with_bias else None
    ref = _fsum_logits(x, router, bias)
    got = (cpp.router_logits(x, router, bias, nthreads=3) if impl == "cpp"
           else moe.router_logits(x.astype(np.float64), router, bias))
    assert got.dtype == F32
    # both sum exactly enough that the fp32 result is the fp32 rounding of the exact sum
    # (one ulp of slack for the double rounding fp64 -> fp32)
    ulp = np.spacing(np.abs(ref).astype(F32)).astype(np.float64)
    assert np.all(np.abs(got.astype(np.float64) - ref) <= ulp), np.max(np.abs(got - ref) / ulp)


def _textbook_h(wg, wu, x, round32):
    f, d = len(wg), len(x)
    h = []
    for j in range(f):
        g = math.fsum(float(wg[j][i]) * float(x[i]) for i in range(d))
        u = math.fsum(float(wu[j][i]) * float(x[i]) for i in range(d))
        if round32:
            g, u = float(F32(g)), float(F32(u))
        v = g / (1.0 + math.exp(-g)) * u
        h.append(float(F32(v)) if round32 else v)
    return np.array(h)


@pytest.mark.parametrize("impl", ["cpp", "numpy"])
@pytest.mark.parametrize("quant_act", [False, True])
def test_expert_hidden_against_textbook_loops(impl, quant_act):
    rng = np.random.default_rng(32)
    d, f, E = 64, 16, 3
    wg = (rng.standard_normal((E + 1, f, d)) * 0.2).astype(F32)
    wu = (rng.standard_normal((E + 1, f, d)) * 0.2).astype(F32)
    wd = (rng.standard_normal((E + 1, d, f)) * 0.2).astype(F32)
    router = np.zeros((d, E), F32)
    x = nvfp4.bf16_rne(rng.standard_normal((3, d))).astype(F32)
    e = 2
    if impl == "cpp":
        L = cpp.quantize_layer(wg, wu, wd, router, k=1, S=1)
        g32, u32, _ = L.expert_f32(e)
        h, _ = cpp.expert(L, e, x, prefill=quant_act)
    else:
        lw = moe.quantize_layer(wg, wu, wd, router)
        g32, u32, _ = lw.expert(e)
        h = moe.expert_hidden(g32, u32, x.astype(np.float64), quant_act=quant_act)
    for t in range(3):
        xt = x[t]
        if quant_act:   # the activation quantiser is pinned in test_oracle_codec.py
            c, s = nvfp4.quantize_activation(xt[None, :])
            xt = nvfp4.dequantize(c, s, 1.0)[0]
        ref = _textbook_h(g32.tolist(), u32.tolist(), xt.tolist(), round32=(impl == "cpp"))
        if impl == "cpp":
            ulp = np.spacing(np.abs(ref).astype(F32)).astype(np.float64)
            assert np.all(np.abs(h[t] - ref) <= 2 * ulp)
        else:
            assert np.allclose(h[t], ref, rtol=1e-12, atol=1e-300)


@pytest.mark.parametrize("impl", ["cpp", "numpy"])
def test_top_k_brute_force_with_ties(impl):
    rng = np.random.default_rng(33)
    topk = cpp.top_k if impl == "cpp" else moe.top_k
    for E, k in ((16, 2), (8, 3), (6, 6), (5, 1), (9, 4)):
        for _ in range(40):
            logits = rng.integers(-3, 4, size=(2, E)).astype(F32)      # many exact ties
            idx = topk(logits, k)
            for t in range(2):
                best = None
                for sub in itertools.combinations(range(E), k):
                    key = (-sum(float(logits[t, e]) for e in sub), sub)
                    if best is None or key < best:
                        best = key
                assert tuple(sorted(idx[t].tolist())) == best[1]
                vals = logits[t, idx[t]]
                assert np.all(np.diff(vals) <= 0)
                for a in range(k - 1):
                    if vals[a] == vals[a + 1]:
                        assert idx[t, a] < idx[t, a + 1]


@pytest.mark.parametrize("impl", ["cpp", "numpy"])
def test_top_k_signed_zero_and_nan(impl):
    topk = cpp.top_k if impl == "cpp" else moe.top_k
    nan = np.nan
    logits = np.array([[nan, 1.0, -0.0, 0.0, nan, -np.inf, -1.0],
                       [nan, nan, nan, nan, nan, nan, nan],
                       [0.0, -0.0, 0.0, -0.0, 2.0, nan, 0.0]], F32)
    idx = topk(logits, 7)
    assert idx[0].tolist() == [1, 2, 3, 6, 5, 0, 4]     # -0 ties +0 (lower index first), NaN last
    assert idx[1].tolist() == list(range(7))              # all NaN: index order
    assert idx[2].tolist() == [4, 0, 1, 2, 3, 6, 5]


@pytest.mark.parametrize("impl", ["cpp", "numpy"])
def test_combine_weights_equal_renormalised_full_softmax(impl):
    rng = np.random.default_rng(34)
    logits = (rng.standard_normal((40, 256)) * 0.9).astype(F32)
    if impl == "cpp":
        idx = cpp.top_k(logits, 6)
        w = cpp.combine_weights(logits, idx).astype(np.float64)
        tol = 2 ** -23
    else:
        idx = moe.top_k(logits, 6)
        w = moe.combine_weights(logits, idx)
        tol = 1e-13
    full = scipy.special.softmax(logits.astype(np.float64), axis=1)
    sel = np.take_along_axis(full, idx.astype(np.int64), axis=1)
    ref = sel / sel.sum(axis=1, keepdims=True)
    assert np.allclose(w, ref, rtol=tol, atol=0)
    assert np.all(np.abs(w.sum(axis=1) - 1) < 6 * tol)


@pytest.mark.parametrize("impl", ["cpp", "numpy"])
def test_bucket_against_bincount_and_sort(impl):
    rng = np.random.default_rng(35)
    T, k, E = 37, 6, 64
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    counts, offsets, perm = (cpp.bucket if impl == "cpp" else moe.bucket)(idx, E)
    assert np.array_equal(counts, np.bincount(idx.ravel(), minlength=E))
    assert offsets[0] == 0 and offsets[-1] == T * k and np.array_equal(np.diff(offsets), counts)
    flat = idx.ravel()
    assert perm.tolist() == sorted(range(T * k), key=lambda s: (flat[s], s))


# --------------------------------------------------------------------------
# C++ codec
# --------------------------------------------------------------------------
def _torch_e4m3(v):
    return torch.from_numpy(np.asarray(v, F32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_cpp_tables_match_torch_and_definition():
    e2, e4 = cpp.tables()
    ref4 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(e4), np.isnan(ref4))
    assert np.array_equal(e4[~np.isnan(e4)], ref4[~np.isnan(ref4)])
    assert e2.tolist()[:8] == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert np.array_equal(e2[8:], -e2[:8])


def test_cpp_e4m3_encode_matches_torch():
    grid = nvfp4.E4M3_TABLE[:0x7F]
    mids = ((grid[:-1] + grid[1:]) / 2).astype(F32)
    rng = np.random.default_rng(36)
    rnd = np.concatenate([rng.uniform(0, 464, 20000), 2.0 ** rng.uniform(-12, 8.8, 20000)]).astype(F32)
    rnd = rnd[rnd <= 464]
    for v in (grid.astype(F32), mids, np.nextafter(mids, F32(np.inf)), np.nextafter(mids, F32(0)), rnd):
        assert np.array_equal(cpp.e4m3_encode(v), _torch_e4m3(v))
    assert np.all(cpp.e4m3_encode(np.array([448, 464.01, 1e6, 3e38], F32)) == 0x7E)


def test_cpp_e2m1_encode_brute_force():
    mags = nvfp4.E2M1_TABLE[:8]
    mids = (mags[:-1] + mags[1:]) / 2
    pts = np.concatenate([mags, mids, np.nextafter(mids, 0), np.nextafter(mids, 10), [5.999, 6.0, 6.5, 100.0]])
    pts = np.concatenate([pts, -pts, [-0.0, -0.2], np.random.default_rng(37).uniform(-8, 8, 4000)]).astype(F32)
    ref = []
    for x in pts.astype(np.float64):
        cands = [(abs(min(max(x, -6.0), 6.0) - nvfp4.E2M1_TABLE[c]), (c & 7) % 2, c)
                 for c in range(16) if not ((c & 8) and nvfp4.E2M1_TABLE[c] == 0)]
        ref.append(min(cands)[2])
    assert np.array_equal(cpp.e2m1_encode(pts), np.array(ref, np.uint8))


def test_cpp_bf16_matches_torch():
    rng = np.random.default_rng(38)
    v = np.concatenate([rng.standard_normal(50000) * 10.0 ** rng.uniform(-30, 30, 50000),
                        [0.0, -0.0, 3.3e38, -3.4e38, 1e-40]]).astype(F32)
    ref = torch.from_numpy(v).to(torch.bfloat16).float().numpy()
    assert np.array_equal(cpp.bf16_rne(v), ref)


@pytest.mark.parametrize("kind", ["normal", "wide", "zero"])
def test_cpp_quantizer_equals_numpy_quantizer(kind):
    rng = np.random.default_rng(39)
    if kind == "normal":
        w = (rng.standard_normal((3, 40, 256)) * 0.02).astype(F32)
    elif kind == "wide":
        w = (rng.standard_normal((2, 16, 512)) * np.logspace(-6, 3, 512)).astype(F32)
    else:
        w = np.zeros((1, 8, 64), F32)
    c, s, ts = cpp.quantize(w, nthreads=2)
    for e in range(w.shape[0]):
        rc, rs, rts = nvfp4.quantize(w[e])
        assert ts[e] == rts and np.array_equal(s[e], rs) and np.array_equal(c[e], rc)
    a = (rng.standard_normal((5, 128)) * 3).astype(F32)
    ca, sa = cpp.quantize_activation(a)
    ra, rsa = nvfp4.quantize_activation(a)
    assert np.array_equal(ca, ra) and np.array_equal(sa, rsa)
    assert np.array_equal(cpp.dequantize(c[0], s[0], ts[0]), nvfp4.dequantize(c[0], s[0], ts[0]).astype(F32))


# --------------------------------------------------------------------------
# C++ layer invariants
# --------------------------------------------------------------------------
def _tiny(rng, d=32, f=16, E=8, S=1, k=2, bias=None):
    n = E + S
    wg = (rng.standard_normal((n, f, d)) * 0.2).astype(F32)
    wu = (rng.standard_normal((n, f, d)) * 0.2).astype(F32)
    wd = (rng.standard_normal((n, d, f)) * 0.2).astype(F32)
    router = (rng.standard_normal((d, E)) * 0.2).astype(F32)
    return cpp.quantize_layer(wg, wu, wd, router, bias, k=k, S=S)


def test_cpp_one_hot_router_reproduces_dense_expert():
    rng = np.random.default_rng(40)
    E, target = 8, 5
    bias = np.full(E, -1e4, F32)
    bias[target] = 1e4
    L = _tiny(rng, E=E, S=0, k=1, bias=bias)
    x = nvfp4.bf16_rne(rng.standard_normal((3, 32))).astype(F32)
    r = cpp.moe_layer(L, x)
    assert np.all(r.idx[:, 0] == target) and np.all(r.w == 1.0)
    wg, wu, wd = (m.tolist() for m in L.expert_f32(target))
    for t in range(3):
        h = _textbook_h(wg, wu, x[t].tolist(), round32=True)
        ref = [math.fsum(wd[r_][j] * h[j] for j in range(len(h))) for r_ in range(32)]
        ulp = np.spacing(np.abs(np.array(ref)).astype(F32)).astype(np.float64)
        assert np.all(np.abs(r.y[t] - ref) <= 2 * ulp)


def test_cpp_k_equals_e_with_equal_logits_gives_mean_plus_shared():
    rng = np.random.default_rng(41)
    E = 6
    L = _tiny(rng, E=E, S=1, k=E)
    L.router[:] = 0
    x = nvfp4.bf16_rne(rng.standard_normal((2, 32))).astype(F32)
    r = cpp.moe_layer(L, x)
    assert np.all(r.w == F32(1.0 / E))
    ref = sum(cpp.expert(L, e, x)[1].astype(np.float64) for e in range(E)) * float(F32(1.0 / E))
    ref = ref + cpp.expert(L, E, x)[1]
    assert np.allclose(r.y, ref, rtol=1e-6, atol=1e-7)


def test_cpp_identical_experts_give_expert_plus_shared():
    rng = np.random.default_rng(42)
    L = _tiny(rng, E=8, S=1, k=3)
    for m in (L.gate, L.up, L.down):
        m[0][:8] = m[0][0]
        m[1][:8] = m[1][0]
        m[2][:8] = m[2][0]
    x = nvfp4.bf16_rne(rng.standard_normal((4, 32))).astype(F32)
    r = cpp.moe_layer(L, x)
    ref = cpp.expert(L, 0, x)[1].astype(np.float64) + cpp.expert(L, 8, x)[1]
    assert np.allclose(r.y, ref, rtol=1e-6, atol=1e-7)


def test_cpp_results_do_not_depend_on_thread_count():
    rng = np.random.default_rng(43)
    L = _tiny(rng, d=64, f=32, E=16, k=4)
    x = nvfp4.bf16_rne(rng.standard_normal((21, 64))).astype(F32)
    for prefill in (False, True):
        a = cpp.moe_layer(L, x, prefill=prefill, nthreads=1)
        b = cpp.moe_layer(L, x, prefill=prefill, nthreads=7)
        assert np.array_equal(a.y, b.y) and np.array_equal(a.idx, b.idx) and np.array_equal(a.logits, b.logits)


@pytest.mark.parametrize("prefill", [False, True])
def test_cpp_layer_agrees_with_numpy_oracle(prefill):
    rng = np.random.default_rng(44)
    d, f, E, S, k = 128, 64, 16, 1, 3
    n = E + S
    wg = (rng.standard_normal((n, f, d)) * 0.02).astype(F32)
    wu = (rng.standard_normal((n, f, d)) * 0.02).astype(F32)
    wd = (rng.standard_normal((n, d, f)) * 0.02).astype(F32)
    router = (rng.standard_normal((d, E)) * 0.02).astype(F32)
    bias = (rng.standard_normal(E) * 0.1).astype(F32)
    L = cpp.quantize_layer(wg, wu, wd, router, bias, k=k, S=S)
    lw = moe.quantize_layer(wg, wu, wd, router, bias)
    x = nvfp4.bf16_rne(rng.standard_normal((29, d))).astype(F32)
    a = cpp.moe_layer(L, x, prefill=prefill)
    b = moe.moe_layer(lw, x.astype(np.float64), k, S, prefill=prefill)
    assert np.array_equal(a.idx, b.idx) and np.array_equal(a.counts, b.counts)
    assert np.allclose(a.w, b.w, rtol=3e-7, atol=0)
    rel = np.linalg.norm(a.y - b.y) / np.linalg.norm(b.y)
    assert rel < (1e-6 if not prefill else 1e-5), rel


# --------------------------------------------------------------------------
# output layer and dense FFN (C++ oracle)
# --------------------------------------------------------------------------
def test_cpp_gemv_against_fsum_loops():
    rng = np.random.default_rng(45)
    w = (rng.standard_normal((24, 64)) * 0.1).astype(F32)
    c, s, ts = cpp.quantize(w)
    wq = cpp.dequantize(c, s, ts).astype(np.float64)
    x = nvfp4.bf16_rne(rng.standard_normal((3, 64))).astype(F32)
    got = cpp.gemv(c, s, ts, x, nthreads=3)
    for t in range(3):
        for r in range(24):
            ref = math.fsum(float(wq[r, k]) * float(x[t, k]) for k in range(64))
            assert abs(float(got[t, r]) - ref) <= float(np.spacing(F32(abs(ref))))


def test_cpp_dense_ffn_against_textbook_loops():
    rng = np.random.default_rng(46)
    d, f = 32, 48
    mats = [cpp.quantize((rng.standard_normal(shape) * 0.2).astype(F32)) for shape in ((f, d), (f, d), (d, f))]
    x = nvfp4.bf16_rne(rng.standard_normal((2, d))).astype(F32)
    y = cpp.dense_ffn(mats[0], mats[1], mats[2], x)
    wg, wu, wd = (cpp.dequantize(*m).tolist() for m in mats)
    for t in range(2):
        h = _textbook_h(wg, wu, x[t].tolist(), round32=True)
        ref = np.array([math.fsum(wd[r][j] * h[j] for j in range(f)) for r in range(d)])
        ulp = np.spacing(np.abs(ref).astype(F32)).astype(np.float64)
        assert np.all(np.abs(y[t] - ref) <= 2 * ulp)
