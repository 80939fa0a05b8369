"""NVFP4 codec and quantiser, written from the format's definition (oracle side).

The Flint pages name NVFP4 as the shipped weight format ("Recursive Flint
40B-A2.5B：まず速さを第一に考えて作られたコーディングモデル", section
"量子化のレシピは最も転用しやすい部分です"; workwonders.jp page, section
"量子化と専用カーネルの最適化") but do not define it.  The reading taken here:

* a value is an E2M1 code (1 sign, 2 exponent bits with bias 1, 1 mantissa
  bit; magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6), two codes per byte with the
  even K index in the low nibble;
* each run of 16 consecutive elements along K carries one E4M3 scale byte
  (OCP E4M3FN: bias 7, subnormals, no infinity, 0x7F/0xFF are NaN, max 448);
* each (expert, matrix) tensor carries one FP32 scale ``ts``;
* the real value is  e2m1(code) * e4m3(scale) * ts  (exact in fp64).

Quantiser (not on the pages; plainest reading, all steps in IEEE fp32 with
round-to-nearest-even, exactly as listed, so both implementations take the
same integer decisions):

    ts   = amax(|W|) / 2688                       (2688 = 6 * 448)
    s_b  = E4M3_rne_satfinite(amax_b / (6 * ts))  (6 * ts rounded first)
    d_b  = e4m3(s_b) * ts
    q    = E2M1_rne_satfinite(w / d_b)            (0 when d_b == 0)

A zero tensor gets ts = 0, all scales 0, all codes 0.  Zero codes are
canonical: a negative value that rounds to magnitude 0 gets code 0, not 8.
Activations (prefill) use the same block step with ts fixed at 1.
"""
from __future__ import annotations

import numpy as np

F32 = np.float32


# --------------------------------------------------------------------------
# decode tables, from the minifloat definitions
# --------------------------------------------------------------------------
def _e2m1_value(code: int) -> float:
    s, e, m = (code >> 3) & 1, (code >> 1) & 3, code & 1
    mag = (m * 0.5) if e == 0 else (2.0 ** (e - 1)) * (1.0 + m / 2.0)
    return -mag if s else mag


def _e4m3_value(code: int) -> float:
    s, e, m = (code >> 7) & 1, (code >> 3) & 15, code & 7
    if e == 15 and m == 7:
        return float("nan")
    mag = (2.0 ** -6) * (m / 8.0) if e == 0 else (2.0 ** (e - 7)) * (1.0 + m / 8.0)
    return -mag if s else mag


#: value of every E2M1 code 0..15 (fp64)
E2M1_TABLE = np.array([_e2m1_value(c) for c in range(16)], dtype=np.float64)
#: value of every E4M3 code 0..255 (fp64; NaN at 0x7F and 0xFF)
E4M3_TABLE = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)

_E2M1_POS = E2M1_TABLE[:8]          # codes 0..7, strictly increasing
_E4M3_POS = E4M3_TABLE[:0x7F]       # codes 0x00..0x7E, strictly increasing


def e2m1_decode(codes) -> np.ndarray:
    return E2M1_TABLE[np.asarray(codes, dtype=np.int64) & 15]


def e4m3_decode(codes) -> np.ndarray:
    return E4M3_TABLE[np.asarray(codes, dtype=np.int64) & 255]


# --------------------------------------------------------------------------
# round-to-nearest-even onto a sorted grid of non-negative values
# --------------------------------------------------------------------------
def _rne_onto_grid(v: np.ndarray, grid: np.ndarray) -> np.ndarray:
    """Code (index into ``grid``) nearest to each v >= 0; ties go to the even code.

    Values at or above the last grid point saturate to it (satfinite).  The
    comparison against the midpoint of the two neighbours is exact: v is an
    fp32 value held in fp64 and every midpoint has few significant bits.
    """
    v = np.asarray(v, dtype=np.float64)
    top = len(grid) - 1
    lo = np.searchsorted(grid, v, side="right") - 1      # grid[lo] <= v
    lo = np.clip(lo, 0, top)
    hi = np.minimum(lo + 1, top)
    mid = (grid[lo] + grid[hi]) / 2.0
    pick_hi = (v > mid) | ((v == mid) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(v >= grid[top], top, code)
    return code.astype(np.int64)


def e4m3_encode(v) -> np.ndarray:
    """E4M3 code of v >= 0 (fp32 input), RNE with saturation at 448."""
    v = np.asarray(v, dtype=F32)
    if np.any(v < 0) or np.any(np.isnan(v)):
        raise ValueError("e4m3_encode expects non-negative finite values")
    return _rne_onto_grid(v, _E4M3_POS).astype(np.uint8)


def e2m1_encode(v) -> np.ndarray:
    """E2M1 code of v (fp32 input), RNE with saturation at +-6, canonical zero."""
    v = np.asarray(v, dtype=F32)
    mag = _rne_onto_grid(np.abs(v), _E2M1_POS)
    sign = (v < 0) & (mag != 0)
    return (mag | (sign.astype(np.int64) << 3)).astype(np.uint8)


# --------------------------------------------------------------------------
# nibble packing: two codes per byte, even K index in the low nibble
# --------------------------------------------------------------------------
def pack_codes(codes: np.ndarray) -> np.ndarray:
    codes = np.asarray(codes, dtype=np.uint8)
    assert codes.shape[-1] % 2 == 0
    return (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)


def unpack_codes(packed: np.ndarray) -> np.ndarray:
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = packed & 15
    out[..., 1::2] = packed >> 4
    return out


# --------------------------------------------------------------------------
# quantiser
# --------------------------------------------------------------------------
def tensor_scale(w: np.ndarray) -> np.float32:
    """ts = amax(|W|) / (6 * 448), one IEEE fp32 division."""
    amax = F32(np.max(np.abs(np.asarray(w, dtype=F32)))) if np.size(w) else F32(0)
    return F32(amax / F32(2688.0))


def quantize_blocks(w: np.ndarray, ts) -> tuple[np.ndarray, np.ndarray]:
    """Block step of the quantiser for a given tensor scale.

    w: fp32 [..., K] with K % 16 == 0.  Returns (packed codes [..., K/2] uint8,
    scale codes [..., K/16] uint8).
    """
    w = np.asarray(w, dtype=F32)
    ts = F32(ts)
    K = w.shape[-1]
    if K % 16:
        raise ValueError("K must be a multiple of 16")
    blocks = w.reshape(w.shape[:-1] + (K // 16, 16))
    if ts == 0:
        z = np.zeros(blocks.shape[:-1], dtype=np.uint8)
        return np.zeros(w.shape[:-1] + (K // 2,), np.uint8), z
    amax_b = np.max(np.abs(blocks), axis=-1).astype(F32)
    six_ts = F32(F32(6.0) * ts)
    s_code = e4m3_encode((amax_b / six_ts).astype(F32))
    d = (e4m3_decode(s_code).astype(F32) * ts).astype(F32)
    safe = np.where(d > 0, d, F32(1.0)).astype(F32)
    q = e2m1_encode((blocks / safe[..., None]).astype(F32))
    q = np.where((d > 0)[..., None], q, np.uint8(0)).astype(np.uint8)
    return pack_codes(q.reshape(w.shape)), s_code


def quantize(w: np.ndarray):
    """Quantise one fp32 weight tensor [rows, K] to NVFP4: (codes, scales, ts)."""
    ts = tensor_scale(w)
    codes, scales = quantize_blocks(w, ts)
    return codes, scales, ts


def quantize_activation(a: np.ndarray):
    """Prefill activation quantiser: the block step with the tensor scale fixed at 1."""
    return quantize_blocks(np.asarray(a, dtype=F32), F32(1.0))


def dequantize(codes: np.ndarray, scales: np.ndarray, ts) -> np.ndarray:
    """Exact real values e2m1 * e4m3 * ts of an NVFP4 tensor, as fp64 [..., K]."""
    q = e2m1_decode(unpack_codes(codes))
    s = e4m3_decode(scales)
    K = q.shape[-1]
    v = q.reshape(q.shape[:-1] + (K // 16, 16)) * s[..., None]
    return v.reshape(q.shape) * np.float64(F32(ts))


# --------------------------------------------------------------------------
# bf16 rounding of fp64 results
# --------------------------------------------------------------------------
def bf16_rne(v) -> np.ndarray:
    """Round fp64 values to the nearest bfloat16 (ties to even); returns fp64.

    bf16 keeps 8 significant bits and fp32's exponent range.  Overflow goes to
    +-inf, values below the smallest subnormal (2^-133) to zero.
    """
    v = np.asarray(v, dtype=np.float64)
    out = np.zeros_like(v)
    fin = np.isfinite(v) & (v != 0)
    vf = v[fin]
    _, e = np.frexp(vf)                          # vf = m * 2^e, 0.5 <= |m| < 1
    e = np.maximum(e, -125)                      # below 2^-126 the quantum stays 2^-133
    q = np.rint(np.ldexp(vf, 8 - e))             # vf / quantum, rounded half to even
    r = np.ldexp(q, e - 8)
    r = np.where(np.abs(r) > 3.3895313892515355e38, np.copysign(np.inf, r), r)
    out[fin] = r
    out[~np.isfinite(v)] = v[~np.isfinite(v)]
    return out
