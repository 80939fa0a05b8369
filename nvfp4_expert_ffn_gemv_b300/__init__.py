"""Python binding of the NVFP4 sparse-MoE FFN library (libnvfp4moe.so, sm_103a).

Argument marshalling only: every function here forwards to the C entry point
of the same name in ``include/nvfp4_moe.h`` with tensors turned into device
pointers, and raises :class:`MoEError` when the call returns a non-zero status.
All computation happens in the library's CUDA kernels; there is no CPU or
PyTorch fallback, and importing this package fails loudly when the library
has not been built (``python nvfp4_expert_ffn_gemv_b300/build.py``).

PyTorch provides device memory and streams only.  ``stream=None`` means
torch's current stream on the tensor's device.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
#: the in-tree library; NVFP4_MOE_LIB may point at another build of the same ABI
LIB_PATH = os.environ.get("NVFP4_MOE_LIB") or os.path.join(_HERE, "libnvfp4moe.so")

MOE_OK = 0
MOE_W_NVFP4 = 0
MOE_W_BF16 = 1
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_OOM",
                4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT", 6: "MOE_ERR_DEVICE_CHECK"}

#: every symbol the C header declares
EXPORTS = ("moe_init", "moe_route", "moe_route_noalloc", "moe_forward_decode", "moe_forward_prefill", "moe_quantize_nvfp4",
           "moe_debug_prefill_h", "moe_debug_routing", "moe_set_profile_events", "moe_set_debug", "moe_debug_logits",
           "moe_debug_wait_selftest", "moe_debug_fail_alloc", "moe_head_init", "moe_head_forward", "moe_ffn_init",
           "moe_ffn_forward", "moe_dense_get_device_status", "moe_dense_kernels_per_forward", "moe_dense_destroy",
           "moe_get_device_status",
           "moe_kernels_per_forward", "moe_destroy", "moe_status_string")
MOE_DEBUG_KEEP_LOGITS = 1
MOE_DEBUG_FORCE_TIMEOUT = 2


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {STATUS_NAMES.get(status, status)} ({status_string(status)})")


class moe_config(ctypes.Structure):
    _fields_ = [("d_model", ctypes.c_int), ("n_experts", ctypes.c_int), ("top_k", ctypes.c_int),
                ("d_ff", ctypes.c_int), ("n_shared", ctypes.c_int), ("d_ff_shared", ctypes.c_int),
                ("max_tokens", ctypes.c_int), ("weight_format", ctypes.c_int)]


class moe_matrix(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("tensor_scale", ctypes.c_void_p), ("bf16", ctypes.c_void_p)]


class moe_weights(ctypes.Structure):
    _fields_ = [("router", ctypes.c_void_p), ("router_bias", ctypes.c_void_p),
                ("gate", moe_matrix), ("up", moe_matrix), ("down", moe_matrix),
                ("shared_gate", moe_matrix), ("shared_up", moe_matrix), ("shared_down", moe_matrix)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python nvfp4_expert_ffn_gemv_b300/build.py` (nvcc, sm_103a)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i, p = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER
    sig = {
        "moe_init": (i, [p(moe_config), p(moe_weights), i, p(vp)]),
        "moe_route": (i, [vp, vp, i, vp, vp, vp, vp]),
        "moe_route_noalloc": (i, [vp, i, vp, vp, i, i, i, vp, vp, vp]),
        "moe_forward_decode": (i, [vp, vp, i, vp, i, vp]),
        "moe_forward_prefill": (i, [vp, vp, i, vp, i, vp]),
        "moe_quantize_nvfp4": (i, [vp, i, i, i, vp, vp, vp, vp]),
        "moe_debug_prefill_h": (i, [vp, i, vp, vp, vp]),
        "moe_debug_routing": (i, [vp, i, vp, vp, vp]),
        "moe_set_profile_events": (i, [vp, vp, vp]),
        "moe_set_debug": (i, [vp, i]),
        "moe_debug_logits": (i, [vp, i, vp, vp]),
        "moe_debug_wait_selftest": (i, [vp, i, vp]),
        "moe_debug_fail_alloc": (i, [i]),
        "moe_head_init": (i, [i, i, p(moe_matrix), i, i, p(vp)]),
        "moe_head_forward": (i, [vp, vp, i, vp, vp]),
        "moe_ffn_init": (i, [i, i, p(moe_matrix), p(moe_matrix), p(moe_matrix), i, i, p(vp)]),
        "moe_ffn_forward": (i, [vp, vp, i, vp, i, vp]),
        "moe_dense_get_device_status": (i, [vp]),
        "moe_dense_kernels_per_forward": (i, [vp, i]),
        "moe_dense_destroy": (i, [vp]),
        "moe_get_device_status": (i, [vp]),
        "moe_kernels_per_forward": (i, [vp, i, i]),
        "moe_destroy": (i, [vp]),
        "moe_status_string": (ctypes.c_char_p, [i]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    return lib


_lib = _load()


def status_string(status: int) -> str:
    return _lib.moe_status_string(int(status)).decode()


def _check(fn: str, status: int) -> None:
    if status != MOE_OK:
        raise MoEError(fn, status)


def _ptr(t):
    """Device (or host) address of a tensor, None/0 for NULL."""
    if t is None:
        return None
    if isinstance(t, int):
        return t or None
    if not t.is_contiguous():
        raise ValueError("tensors passed to the library must be contiguous")
    return t.data_ptr()


def _stream(stream, device=None):
    import torch
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _matrix(m):
    """dict(codes=, scales=, tensor_scale=) or dict(bf16=) -> moe_matrix."""
    m = m or {}
    return moe_matrix(_ptr(m.get("codes")), _ptr(m.get("scales")), _ptr(m.get("tensor_scale")),
                      _ptr(m.get("bf16")))


def moe_init(cfg: dict, weights: dict, device: int = 0):
    """Create a layer context.  ``cfg`` has the moe_config fields; ``weights`` has
    router, router_bias (optional) and gate/up/down/shared_gate/shared_up/shared_down
    dicts of tensors (host or device).  Returns an opaque handle (int)."""
    c = moe_config(cfg["d_model"], cfg["n_experts"], cfg["top_k"], cfg["d_ff"], cfg.get("n_shared", 1),
                   cfg.get("d_ff_shared", cfg["d_ff"]), cfg["max_tokens"],
                   cfg.get("weight_format", MOE_W_NVFP4))
    w = moe_weights(_ptr(weights["router"]), _ptr(weights.get("router_bias")),
                    *(_matrix(weights.get(k)) for k in
                      ("gate", "up", "down", "shared_gate", "shared_up", "shared_down")))
    out = ctypes.c_void_p()
    _check("moe_init", _lib.moe_init(ctypes.byref(c), ctypes.byref(w), int(device), ctypes.byref(out)))
    return out.value


def moe_route(ctx, x, T: int, idx=None, w=None, counts=None, stream=None) -> None:
    _check("moe_route", _lib.moe_route(ctx, _ptr(x), int(T), _ptr(idx), _ptr(w), _ptr(counts),
                                       _stream(stream)))


def moe_route_noalloc(x, T: int, router, router_bias, d_model: int, n_experts: int, top_k: int, idx, w,
                      stream=None) -> None:
    _check("moe_route_noalloc", _lib.moe_route_noalloc(_ptr(x), int(T), _ptr(router), _ptr(router_bias),
                                                       int(d_model), int(n_experts), int(top_k), _ptr(idx),
                                                       _ptr(w), _stream(stream)))


def moe_forward_decode(ctx, x, T: int, y, residual: int = 0, stream=None) -> None:
    _check("moe_forward_decode", _lib.moe_forward_decode(ctx, _ptr(x), int(T), _ptr(y), int(residual),
                                                         _stream(stream)))


def moe_forward_prefill(ctx, x, T: int, y, residual: int = 0, stream=None) -> None:
    _check("moe_forward_prefill", _lib.moe_forward_prefill(ctx, _ptr(x), int(T), _ptr(y), int(residual),
                                                           _stream(stream)))


def moe_quantize_nvfp4(w, n: int, rows: int, K: int, codes, scales, ts, stream=None) -> None:
    _check("moe_quantize_nvfp4", _lib.moe_quantize_nvfp4(_ptr(w), int(n), int(rows), int(K), _ptr(codes),
                                                         _ptr(scales), _ptr(ts), _stream(stream)))


def moe_debug_prefill_h(ctx, T: int, h_codes, h_scales, stream=None) -> None:
    _check("moe_debug_prefill_h", _lib.moe_debug_prefill_h(ctx, int(T), _ptr(h_codes), _ptr(h_scales),
                                                           _stream(stream)))


def moe_debug_routing(ctx, T: int, idx, w, stream=None) -> None:
    _check("moe_debug_routing", _lib.moe_debug_routing(ctx, int(T), _ptr(idx), _ptr(w), _stream(stream)))


def moe_set_profile_events(ctx, start=None, stop=None) -> None:
    ev = lambda e: None if e is None else (e if isinstance(e, int) else e.cuda_event)  # noqa: E731
    _check("moe_set_profile_events", _lib.moe_set_profile_events(ctx, ev(start), ev(stop)))


def moe_set_debug(ctx, flags: int) -> None:
    _check("moe_set_debug", _lib.moe_set_debug(ctx, int(flags)))


def moe_debug_logits(ctx, T: int, logits, stream=None) -> None:
    _check("moe_debug_logits", _lib.moe_debug_logits(ctx, int(T), _ptr(logits), _stream(stream)))


def moe_debug_wait_selftest(ctx, spin_limit: int, stream=None) -> None:
    _check("moe_debug_wait_selftest", _lib.moe_debug_wait_selftest(ctx, int(spin_limit), _stream(stream)))


def moe_debug_fail_alloc(n: int) -> None:
    _check("moe_debug_fail_alloc", _lib.moe_debug_fail_alloc(int(n)))


def moe_head_init(vocab: int, d_model: int, w: dict, max_tokens: int, device: int = 0):
    """lm_head context from w = dict(codes=, scales=, tensor_scale=) (host or device tensors)."""
    out = ctypes.c_void_p()
    m = _matrix(w)
    _check("moe_head_init", _lib.moe_head_init(int(vocab), int(d_model), ctypes.byref(m), int(max_tokens),
                                               int(device), ctypes.byref(out)))
    return out.value


def moe_head_forward(ctx, x, T: int, logits, stream=None) -> None:
    _check("moe_head_forward", _lib.moe_head_forward(ctx, _ptr(x), int(T), _ptr(logits), _stream(stream)))


def moe_ffn_init(d_model: int, d_ff: int, gate: dict, up: dict, down: dict, max_tokens: int, device: int = 0):
    """Dense SwiGLU FFN context from NVFP4 gate/up/down dicts (codes, scales, tensor_scale)."""
    out = ctypes.c_void_p()
    g, u, d = _matrix(gate), _matrix(up), _matrix(down)
    _check("moe_ffn_init", _lib.moe_ffn_init(int(d_model), int(d_ff), ctypes.byref(g), ctypes.byref(u),
                                             ctypes.byref(d), int(max_tokens), int(device), ctypes.byref(out)))
    return out.value


def moe_ffn_forward(ctx, x, T: int, y, residual: int = 0, stream=None) -> None:
    _check("moe_ffn_forward", _lib.moe_ffn_forward(ctx, _ptr(x), int(T), _ptr(y), int(residual), _stream(stream)))


def moe_dense_get_device_status(ctx) -> int:
    return int(_lib.moe_dense_get_device_status(ctx))


def moe_dense_kernels_per_forward(ctx, T: int) -> int:
    return int(_lib.moe_dense_kernels_per_forward(ctx, int(T)))


def moe_dense_destroy(ctx) -> None:
    _check("moe_dense_destroy", _lib.moe_dense_destroy(ctx))


def moe_get_device_status(ctx) -> int:
    """Synchronise and return (then clear) the device status word; 0 = MOE_OK."""
    return int(_lib.moe_get_device_status(ctx))


def moe_kernels_per_forward(ctx, T: int, prefill: int = 0) -> int:
    return int(_lib.moe_kernels_per_forward(ctx, int(T), int(prefill)))


def moe_destroy(ctx) -> None:
    _check("moe_destroy", _lib.moe_destroy(ctx))


def moe_status_string(status: int) -> str:
    return status_string(status)


# ---------------------------------------------------------------------------
# marshalling helpers built on the entry points above
# ---------------------------------------------------------------------------
def quantize(w, stream=None):
    """NVFP4-quantise a CUDA fp32 tensor [n, rows, K] (or [rows, K]) with the library's
    kernel.  Returns (codes uint8 [..., K/2], scales uint8 [..., K/16], ts fp32 [n])."""
    import torch
    squeeze = w.dim() == 2
    w3 = w.unsqueeze(0) if squeeze else w
    n, rows, K = w3.shape
    codes = torch.empty((n, rows, K // 2), dtype=torch.uint8, device=w.device)
    scales = torch.empty((n, rows, K // 16), dtype=torch.uint8, device=w.device)
    ts = torch.empty((n,), dtype=torch.float32, device=w.device)
    moe_quantize_nvfp4(w3.contiguous(), n, rows, K, codes, scales, ts, stream)
    if squeeze:
        return codes[0], scales[0], ts
    return codes, scales, ts
