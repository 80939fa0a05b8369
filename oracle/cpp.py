"""ctypes front end of the C++ oracle (moe_oracle.cpp) -- TEST INFRASTRUCTURE ONLY.

The C++ oracle is the plain CPU reference the CUDA library is checked
against: NVFP4 dequantised to FP32, every value between steps an FP32 number,
each dot product summed in FP64 in index order and rounded once to FP32 (the
definitions are at the top of moe_oracle.cpp).  This module builds it with
g++ (no fast-math, no FMA contraction) into ``oracle/liboracle.so`` when the
library is missing or older than its source, and wraps every entry point for
numpy arrays.  It shares no code with the CUDA path.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_oracle.cpp")
LIB = os.path.join(HERE, "liboracle.so")
CXX = os.environ.get("CXX", "g++")
FLAGS = ["-O2", "-std=c++17", "-fPIC", "-shared", "-pthread", "-ffp-contract=off", "-fno-fast-math"]

F32 = np.float32
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile moe_oracle.cpp into liboracle.so (if missing, stale or forced)."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + f".{os.getpid()}.tmp"
    r = subprocess.run([CXX, *FLAGS, "-o", tmp, SRC], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"building the C++ oracle failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


class _Matrix(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("ts", ctypes.c_void_p)]


class _Layer(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int), ("E", ctypes.c_int), ("k", ctypes.c_int), ("f", ctypes.c_int),
                ("S", ctypes.c_int), ("router", ctypes.c_void_p), ("bias", ctypes.c_void_p),
                ("gate", _Matrix), ("up", _Matrix), ("down", _Matrix),
                ("dense_gate", ctypes.c_void_p), ("dense_up", ctypes.c_void_p), ("dense_down", ctypes.c_void_p)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            vp, i, lg = ctypes.c_void_p, ctypes.c_int, ctypes.c_long
            sig = {
                "or_tables": [vp, vp],
                "or_e4m3_encode": [vp, lg, vp],
                "or_e2m1_encode": [vp, lg, vp],
                "or_quantize": [vp, i, i, i, vp, vp, vp, i],
                "or_quantize_act": [vp, i, i, vp, vp],
                "or_dequantize": [vp, vp, ctypes.c_float, i, i, vp],
                "or_bf16_rne": [vp, lg, vp],
                "or_router_logits": [vp, i, i, vp, vp, i, vp, i],
                "or_top_k": [vp, i, i, i, vp],
                "or_combine_weights": [vp, vp, i, i, i, vp],
                "or_bucket": [vp, i, i, i, vp, vp, vp],
                "or_expert": [ctypes.POINTER(_Layer), i, vp, i, i, vp, vp, i],
                "or_moe_layer": [ctypes.POINTER(_Layer), vp, i, i, vp, vp, vp, vp, vp, vp, i],
                "or_gemv": [vp, vp, ctypes.c_float, i, i, vp, i, vp, i],
                "or_dense_ffn": [_Matrix, _Matrix, _Matrix, i, i, vp, i, vp, i],
            }
            for name, args in sig.items():
                fn = getattr(L, name)
                fn.restype, fn.argtypes = None, args
            _lib = L
    return _lib


def _c(a, dtype):
    """C-contiguous array of the given dtype (a copy only if needed)."""
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a):
    return None if a is None else a.ctypes.data


# --------------------------------------------------------------------------
# codec
# --------------------------------------------------------------------------
def tables():
    """(E2M1 values of codes 0..15, E4M3 values of codes 0..255) as fp64."""
    e2, e4 = np.zeros(16), np.zeros(256)
    lib().or_tables(_p(e2), _p(e4))
    return e2, e4


def e4m3_encode(v) -> np.ndarray:
    v = _c(v, F32)
    if np.any(v < 0) or np.any(np.isnan(v)):
        raise ValueError("e4m3_encode expects non-negative finite values")
    out = np.empty(v.shape, np.uint8)
    lib().or_e4m3_encode(_p(v), v.size, _p(out))
    return out


def e2m1_encode(v) -> np.ndarray:
    v = _c(v, F32)
    out = np.empty(v.shape, np.uint8)
    lib().or_e2m1_encode(_p(v), v.size, _p(out))
    return out


def quantize(w, nthreads: int = 0):
    """Weight quantiser.  w fp32 [rows, K] or [n, rows, K] -> (codes, scales, ts)."""
    w = _c(w, F32)
    squeeze = w.ndim == 2
    w3 = w[None] if squeeze else w
    n, rows, K = w3.shape
    if K % 16:
        raise ValueError("K must be a multiple of 16")
    codes = np.empty((n, rows, K // 2), np.uint8)
    scales = np.empty((n, rows, K // 16), np.uint8)
    ts = np.empty((n,), F32)
    lib().or_quantize(_p(w3), n, rows, K, _p(codes), _p(scales), _p(ts), nthreads)
    if squeeze:
        return codes[0], scales[0], ts[0]
    return codes, scales, ts


def quantize_activation(a):
    """Activation quantiser (tensor scale 1): a fp32 [rows, K] -> (codes, scales)."""
    a = _c(a, F32)
    rows, K = a.shape
    codes = np.empty((rows, K // 2), np.uint8)
    scales = np.empty((rows, K // 16), np.uint8)
    lib().or_quantize_act(_p(a), rows, K, _p(codes), _p(scales))
    return codes, scales


def dequantize(codes, scales, ts) -> np.ndarray:
    """fp32 values of one NVFP4 tensor [rows, K]."""
    codes, scales = _c(codes, np.uint8), _c(scales, np.uint8)
    rows, K = codes.shape[0], codes.shape[1] * 2
    out = np.empty((rows, K), F32)
    lib().or_dequantize(_p(codes), _p(scales), float(ts), rows, K, _p(out))
    return out


def bf16_rne(v) -> np.ndarray:
    """fp32 -> nearest bf16 (ties to even), as fp32 values."""
    v = _c(v, F32)
    out = np.empty_like(v)
    lib().or_bf16_rne(_p(v), v.size, _p(out))
    return out


# --------------------------------------------------------------------------
# router
# --------------------------------------------------------------------------
def router_logits(x, router, bias=None, nthreads: int = 0) -> np.ndarray:
    x, router = _c(x, F32), _c(router, F32)
    T, d = x.shape
    E = router.shape[1]
    b = None if bias is None else _c(bias, F32)
    out = np.empty((T, E), F32)
    lib().or_router_logits(_p(x), T, d, _p(router), _p(b), E, _p(out), nthreads)
    return out


def top_k(logits, k: int) -> np.ndarray:
    logits = _c(logits, F32)
    T, E = logits.shape
    idx = np.empty((T, k), np.int32)
    lib().or_top_k(_p(logits), T, E, k, _p(idx))
    return idx


def combine_weights(logits, idx) -> np.ndarray:
    logits, idx = _c(logits, F32), _c(idx, np.int32)
    T, E = logits.shape
    k = idx.shape[1]
    w = np.empty((T, k), F32)
    lib().or_combine_weights(_p(logits), _p(idx), T, E, k, _p(w))
    return w


def bucket(idx, n_experts: int):
    idx = _c(idx, np.int32)
    T, k = idx.shape
    counts = np.empty(n_experts, np.int32)
    offsets = np.empty(n_experts + 1, np.int32)
    perm = np.empty(T * k, np.int32)
    lib().or_bucket(_p(idx), T, k, n_experts, _p(counts), _p(offsets), _p(perm))
    return counts, offsets, perm


# --------------------------------------------------------------------------
# layer
# --------------------------------------------------------------------------
@dataclasses.dataclass
class Layer:
    """One layer's weights (experts 0..E-1 routed, E..E+S-1 shared).

    NVFP4: gate/up codes [n, f, d/2], scales [n, f, d/16], ts [n]; down
    [n, d, f/2], [n, d, f/16], ts [n].  bf16 weights (the tiny configuration):
    ``dense`` = (W_gate [n, f, d], W_up [n, f, d], W_down [n, d, f]) as fp32
    values, gate/up/down None.  router fp32 [d, E]; bias fp32 [E] or None.
    """
    router: np.ndarray
    bias: np.ndarray | None
    gate: tuple | None
    up: tuple | None
    down: tuple | None
    k: int
    S: int = 1
    dense: tuple | None = None

    def __post_init__(self):
        self.router = _c(self.router, F32)
        self.bias = None if self.bias is None else _c(self.bias, F32)
        if self.dense is not None:
            self.dense = tuple(_c(w, F32) for w in self.dense)
            mats = (_Matrix(None, None, None),) * 3
            dense = tuple(_p(w) for w in self.dense)
        else:
            fix = lambda m: (_c(m[0], np.uint8), _c(m[1], np.uint8), _c(m[2], F32))  # noqa: E731
            self.gate, self.up, self.down = fix(self.gate), fix(self.up), fix(self.down)
            mats = tuple(_Matrix(*(_p(a) for a in m)) for m in (self.gate, self.up, self.down))
            dense = (None, None, None)
        self._c = _Layer(self.d, self.E, self.k, self.f, self.S, _p(self.router), _p(self.bias), *mats, *dense)

    @property
    def d(self) -> int:
        return self.router.shape[0]

    @property
    def E(self) -> int:
        return self.router.shape[1]

    @property
    def f(self) -> int:
        return self.dense[0].shape[1] if self.dense is not None else self.gate[0].shape[1]

    def expert_f32(self, e: int):
        """fp32 (W_gate [f, d], W_up [f, d], W_down [d, f]) of expert e."""
        if self.dense is not None:
            return tuple(w[e].copy() for w in self.dense)
        return tuple(dequantize(m[0][e], m[1][e], m[2][e]) for m in (self.gate, self.up, self.down))


def quantize_layer(w_gate, w_up, w_down, router, bias=None, k: int = 6, S: int = 1, experts=None,
                   nthreads: int = 0) -> Layer:
    """NVFP4-quantise fp32 expert weights [n, f, d] / [n, d, f] with the oracle quantiser.

    ``experts`` restricts the work to a subset (the others stay zero).
    """
    w_gate, w_up, w_down = (np.asarray(w, F32) for w in (w_gate, w_up, w_down))
    n = w_gate.shape[0]
    sel = list(range(n)) if experts is None else sorted(set(int(e) for e in experts))

    def q(w):
        codes = np.zeros((n, w.shape[1], w.shape[2] // 2), np.uint8)
        scales = np.zeros((n, w.shape[1], w.shape[2] // 16), np.uint8)
        ts = np.zeros((n,), F32)
        if sel:
            c, s, t = quantize(w[sel], nthreads)
            codes[sel], scales[sel], ts[sel] = c, s, t
        return codes, scales, ts

    return Layer(router=router, bias=bias, gate=q(w_gate), up=q(w_up), down=q(w_down), k=k, S=S)


def expert(layer: Layer, e: int, x, prefill: bool = False, nthreads: int = 0):
    """(h fp32 [T, f] before any activation quantisation, y fp32 [T, d]) of expert e on x [T, d]."""
    x = _c(x, F32)
    T = x.shape[0]
    h = np.empty((T, layer.f), F32)
    y = np.empty((T, layer.d), F32)
    lib().or_expert(ctypes.byref(layer._c), int(e), _p(x), T, int(prefill), _p(h), _p(y), nthreads)
    return h, y


def near_ties(logits, k: int, gap: float = 1e-6) -> np.ndarray:
    """Per token: True where two adjacent logits among the k+1 best differ by less than ``gap``."""
    s = -np.sort(-np.asarray(logits, np.float64), axis=1)[:, : k + 1]
    return np.any(np.abs(np.diff(s, axis=1)) < gap, axis=1)


@dataclasses.dataclass
class LayerResult:
    y: np.ndarray          # fp32 [T, d]
    y_bf16: np.ndarray     # fp32 [T, d], values rounded to bf16
    logits: np.ndarray     # fp32 [T, E]
    idx: np.ndarray        # int32 [T, k]
    w: np.ndarray          # fp32 [T, k]
    counts: np.ndarray     # int32 [E]
    near_tie: np.ndarray   # bool [T]


def moe_layer(layer: Layer, x, prefill: bool = False, force_idx=None, nthreads: int = 0) -> LayerResult:
    """y[t] = sum_j w[t, j] expert_{idx[t, j]}(x_t) + sum_s shared_s(x_t), x fp32 [T, d]."""
    x = _c(x, F32)
    T = x.shape[0]
    E, k = layer.E, layer.k
    y = np.empty((T, layer.d), F32)
    logits = np.empty((T, E), F32)
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), F32)
    counts = np.empty((E,), np.int32)
    fi = None if force_idx is None else _c(force_idx, np.int32)
    lib().or_moe_layer(ctypes.byref(layer._c), _p(x), T, int(prefill), _p(fi), _p(y), _p(logits), _p(idx),
                       _p(w), _p(counts), nthreads)
    return LayerResult(y=y, y_bf16=bf16_rne(y), logits=logits, idx=idx, w=w, counts=counts,
                       near_tie=near_ties(logits, k))


def route(x, router, bias, k: int, nthreads: int = 0) -> LayerResult:
    """The router alone on x fp32 [T, d]: logits, idx, w and counts (y fields are None)."""
    logits = router_logits(x, router, bias, nthreads)
    idx = top_k(logits, k)
    w = combine_weights(logits, idx)
    counts, _, _ = bucket(idx, logits.shape[1])
    return LayerResult(y=None, y_bf16=None, logits=logits, idx=idx, w=w, counts=counts,
                       near_tie=near_ties(logits, k))


def gemv(codes, scales, ts, x, nthreads: int = 0) -> np.ndarray:
    """Output layer: logits fp32 [T, R] = x [T, K] . W^T, W one NVFP4 tensor (codes [R, K/2])."""
    codes, scales, x = _c(codes, np.uint8), _c(scales, np.uint8), _c(x, F32)
    R, K = codes.shape[0], codes.shape[1] * 2
    T = x.shape[0]
    out = np.empty((T, R), F32)
    lib().or_gemv(_p(codes), _p(scales), float(ts), R, K, _p(x), T, _p(out), nthreads)
    return out


def dense_ffn(gate, up, down, x, nthreads: int = 0) -> np.ndarray:
    """Dense SwiGLU FFN: y fp32 [T, d]; gate/up = (codes [f, d/2], scales, ts), down = ([d, f/2], ...)."""
    fix = lambda m: (_c(m[0], np.uint8), _c(m[1], np.uint8), np.array([m[2]], F32).reshape(1))  # noqa: E731
    g, u, dn = fix(gate), fix(up), fix(down)
    x = _c(x, F32)
    T, d = x.shape
    f = g[0].shape[0]
    y = np.empty((T, d), F32)
    mats = [_Matrix(*(_p(a) for a in m)) for m in (g, u, dn)]
    lib().or_dense_ffn(mats[0], mats[1], mats[2], d, f, _p(x), T, _p(y), nthreads)
    return y


def residual(x, y) -> np.ndarray:
    """Next layer input of the stack: bf16_rne(x + y) with the sum in fp32."""
    return bf16_rne((_c(x, F32) + _c(y, F32)).astype(F32))
