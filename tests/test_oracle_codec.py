"""Pins of the oracle's NVFP4 codec against things other than itself.

* E4M3: decode and round-to-nearest-even encode checked against torch's
  float8_e4m3fn conversions (a library routine) on every code, every midpoint
  between neighbouring codes, and random values.
* E2M1: no CPU library converts FP4, so the encoder is checked against a
  brute-force nearest search over all 16 codes, every code must round-trip,
  and every E2M1 magnitude must lie on the E4M3 grid with at most one
  mantissa bit (the two formats share their definition of a minifloat).
* quantiser: closed-form reconstruction bound, saturation of the block that
  holds the tensor maximum, zero handling, and the bit budget of 4.5 bits
  per weight that the page figures support (see test_oracle_pages.py).
* bf16 rounding: against torch's float32 -> bfloat16 conversion, plus
  hand-built fp64 ties.
"""
import numpy as np
import pytest
import torch

from oracle import nvfp4

F32 = np.float32


def _torch_e4m3(v):
    return torch.from_numpy(np.asarray(v, F32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_decode_matches_torch_all_codes():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    ours = nvfp4.E4M3_TABLE
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    assert np.array_equal(ours[~np.isnan(ours)], ref[~np.isnan(ref)])
    assert np.isnan(ours[0x7F]) and np.isnan(ours[0xFF])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9


def test_e4m3_encode_matches_torch_midpoints_and_random():
    grid = nvfp4.E4M3_TABLE[:0x7F]
    mids = ((grid[:-1] + grid[1:]) / 2).astype(F32)
    assert np.array_equal(mids.astype(np.float64), (grid[:-1] + grid[1:]) / 2)  # exact in fp32
    up = np.nextafter(mids, F32(np.inf))
    dn = np.nextafter(mids, F32(0))
    rng = np.random.default_rng(1)
    rnd = np.concatenate([rng.uniform(0, 464, 20000), 2.0 ** rng.uniform(-12, 8.8, 20000)]).astype(F32)
    rnd = rnd[rnd <= 464]
    for v in (grid.astype(F32), mids, up, dn, rnd):
        assert np.array_equal(nvfp4.e4m3_encode(v), _torch_e4m3(v))


def test_e4m3_encode_saturates():
    v = np.array([448, 464, 464.01, 480, 1e6, 3e38], F32)
    assert np.all(nvfp4.e4m3_encode(v) == 0x7E)
    with pytest.raises(ValueError):
        nvfp4.e4m3_encode(np.array([-1.0], F32))


def _e2m1_brute(v):
    """Nearest of the 16 code values by exhaustive search; ties to the even magnitude code."""
    out = []
    for x in np.asarray(v, F32).astype(np.float64):
        best = None
        for c in range(16):
            val = nvfp4.E2M1_TABLE[c]
            if (c & 8) and val == 0:
                continue  # -0 is never produced (canonical zero)
            dist = abs(min(max(x, -6.0), 6.0) - val)
            key = (dist, (c & 7) % 2, c)
            if best is None or key < best[0]:
                best = (key, c)
        out.append(best[1])
    return np.array(out, np.uint8)


def test_e2m1_encode_brute_force():
    mags = nvfp4.E2M1_TABLE[:8]
    mids = (mags[:-1] + mags[1:]) / 2
    pts = np.concatenate([mags, mids, np.nextafter(mids, 0), np.nextafter(mids, 10), [5.999, 6.0, 6.5, 7.0, 100.0, 1e30]])
    pts = np.concatenate([pts, -pts, np.random.default_rng(2).uniform(-8, 8, 4000)]).astype(F32)
    assert np.array_equal(nvfp4.e2m1_encode(pts), _e2m1_brute(pts))
    # the published rounding table of the E2M1 grid (ties to even)
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], F32)
    assert list(nvfp4.e2m1_decode(nvfp4.e2m1_encode(ties))) == [0, 1, 1, 2, 2, 4, 4]


def test_e2m1_roundtrip_every_code_and_grid_relation():
    for c in range(16):
        v = nvfp4.E2M1_TABLE[c]
        back = int(nvfp4.e2m1_encode(np.array([v], F32))[0])
        assert back == (0 if c == 8 else c)
    mags = nvfp4.E2M1_TABLE[1:8]
    assert mags.max() == 6.0 and mags.min() == 0.5 and np.all(np.diff(nvfp4.E2M1_TABLE[:8]) > 0)
    # each E2M1 magnitude is an E4M3 value whose code has only the top mantissa bit
    codes = _torch_e4m3(mags)
    assert np.array_equal(nvfp4.E4M3_TABLE[codes], mags)
    assert np.all((codes & 3) == 0)
    assert np.array_equal(nvfp4.E2M1_TABLE[8:], -nvfp4.E2M1_TABLE[:8])


def test_pack_unpack_low_nibble_is_even_k():
    codes = np.array([[1, 2, 3, 4, 15, 0]], np.uint8)
    packed = nvfp4.pack_codes(codes)
    assert packed.tolist() == [[0x21, 0x43, 0x0F]]
    assert np.array_equal(nvfp4.unpack_codes(packed), codes)


def _grid_gap(mag):
    """Spacing of the E2M1 grid around magnitude |q| (upper neighbour gap)."""
    g = nvfp4.E2M1_TABLE[:8]
    i = np.clip(np.searchsorted(g, mag, side="right") - 1, 0, 6)
    return g[i + 1] - g[i]


def test_quantize_reconstruction_bound():
    rng = np.random.default_rng(3)
    w = (rng.standard_normal((64, 256)) * 0.02).astype(F32)
    w[5, 17] = 0.5   # a tensor maximum far above the rest
    codes, scales, ts = nvfp4.quantize(w)
    assert ts == F32(F32(0.5) / F32(2688))
    deq = nvfp4.dequantize(codes, scales, ts)
    s = nvfp4.e4m3_decode(scales)
    d = np.repeat(s, 16, axis=1) * np.float64(ts)
    # every element lies within half a grid step (in units of d) of its value
    err = np.abs(deq - w.astype(np.float64))
    q = np.abs(deq) / np.where(d > 0, d, 1)
    assert np.all(err <= 0.5 * _grid_gap(np.minimum(q, 4)) * d * (1 + 1e-6) + 1e-30)
    # no element saturated: the block scale makes every |w| / d <= 6 (up to the scale's rounding)
    ratio = np.abs(w.astype(np.float64)) / d
    assert np.all(ratio <= 6.0 * (1 + 2 ** -3))
    # the block holding the tensor maximum gets the largest scale, 448
    assert scales[5, 17 // 16] == 0x7E
    assert abs(deq[5, 17] - 0.5) <= 0.5 * 2 ** -24 * 448 * 6 * float(ts) * 8


def test_quantize_zero_and_exact_values():
    c, s, ts = nvfp4.quantize(np.zeros((2, 32), F32))
    assert ts == 0 and not c.any() and not s.any()
    # amax = 2688 * 2^-12 makes ts = 2^-12 exactly; blocks whose values sit on
    # the E2M1 grid times a representable E4M3 scale then round-trip exactly
    d0 = 448 * 2.0 ** -12
    w = np.zeros((1, 32), F32)
    w[0, :8] = np.array([6, -4, 3, 0.5, -0.5, 1.5, 0, 2]) * d0
    w[0, 16:24] = np.array([6, 1, 2, 3, 4, -6, 0.5, 1]) * (d0 / 4)
    codes, scales, ts = nvfp4.quantize(w)
    assert ts == 2.0 ** -12
    assert scales.tolist() == [[0x7E, 0x6E]]     # 448 and 112
    assert np.array_equal(nvfp4.dequantize(codes, scales, ts), w.astype(np.float64))


def test_quantize_activation_unit_tensor_scale():
    a = np.array([[3.0, -1.5, 0, 0.75] + [0] * 12], F32)   # amax 3 -> scale 0.5 exactly
    c, s = nvfp4.quantize_activation(a)
    assert nvfp4.e4m3_decode(s)[0, 0] == 0.5
    assert np.array_equal(nvfp4.dequantize(c, s, 1.0), a.astype(np.float64))


def test_bf16_rne_matches_torch():
    rng = np.random.default_rng(4)
    v = np.concatenate([rng.standard_normal(50000) * 10.0 ** rng.uniform(-30, 30, 50000),
                        2.0 ** rng.uniform(-140, -120, 2000)]).astype(F32)
    ref = torch.from_numpy(v).to(torch.bfloat16).double().numpy()
    assert np.array_equal(nvfp4.bf16_rne(v.astype(np.float64)), ref)


def test_bf16_rne_fp64_ties_and_edges():
    one_ulp = 2.0 ** -7
    assert nvfp4.bf16_rne(np.array([1 + one_ulp / 2]))[0] == 1.0            # tie to even
    assert nvfp4.bf16_rne(np.array([1 + 3 * one_ulp / 2]))[0] == 1 + 2 * one_ulp
    assert nvfp4.bf16_rne(np.array([1 + one_ulp / 2 + 2 ** -40]))[0] == 1 + one_ulp  # no double rounding
    assert nvfp4.bf16_rne(np.array([3.4e38]))[0] == np.inf
    assert nvfp4.bf16_rne(np.array([0.0, -0.0]))[0] == 0.0
