"""The C-ABI library loads without a GPU, exports every entry point the header
declares, and rejects bad arguments on the host before touching a device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _header_functions():
    src = open(os.path.join(ROOT, "include", "nvfp4_moe.h")).read()
    return set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", src))


def test_library_exports_every_declared_symbol():
    import nvfp4_expert_ffn_gemv_b300 as lib
    declared = _header_functions()
    assert declared == set(lib.EXPORTS)
    raw = ctypes.CDLL(lib.LIB_PATH)
    for name in declared:
        assert hasattr(raw, name), name


def test_status_strings():
    import nvfp4_expert_ffn_gemv_b300 as lib
    assert lib.status_string(0) == "ok"
    assert "argument" in lib.status_string(1)
    assert lib.status_string(99) == "unknown status"


def _cfg(**kw):
    c = dict(d_model=256, n_experts=16, top_k=2, d_ff=128, n_shared=1, d_ff_shared=128, max_tokens=4,
             weight_format=0)
    c.update(kw)
    return c


@pytest.mark.parametrize("bad,code", [
    (dict(d_model=0), 1), (dict(top_k=0), 1), (dict(top_k=17), 1), (dict(max_tokens=0), 1),
    (dict(weight_format=7), 1), (dict(n_shared=-1), 1),
    (dict(d_model=300), 2), (dict(d_ff=96), 2), (dict(n_experts=300, top_k=2), 2), (dict(top_k=9, n_experts=16), 2),
    (dict(d_ff_shared=256), 2), (dict(max_tokens=70000), 2), (dict(d_model=8192), 2),
])
def test_init_rejects_bad_config_on_host(bad, code):
    import nvfp4_expert_ffn_gemv_b300 as lib
    with pytest.raises(lib.MoEError) as ei:
        lib.moe_init(_cfg(**bad), {"router": 0x1000})
    assert ei.value.status == code


def test_init_rejects_missing_weights_on_host():
    import nvfp4_expert_ffn_gemv_b300 as lib
    with pytest.raises(lib.MoEError) as ei:
        lib.moe_init(_cfg(), {"router": None})
    assert ei.value.status == 1
    with pytest.raises(lib.MoEError) as ei:   # NVFP4 format without codes
        lib.moe_init(_cfg(), {"router": 0x1000, "gate": {"bf16": 0x1000}})
    assert ei.value.status == 1


def test_calls_reject_null_context_and_bad_sizes():
    import nvfp4_expert_ffn_gemv_b300 as L
    lib = L._lib
    assert lib.moe_forward_decode(None, 0x1000, 1, 0x2000, 0, None) == 1
    assert lib.moe_forward_prefill(None, 0x1000, 1, 0x2000, 0, None) == 1
    assert lib.moe_route(None, 0x1000, 1, None, None, None, None) == 1
    assert lib.moe_get_device_status(None) == 1
    assert lib.moe_set_profile_events(None, None, None) == 1
    assert lib.moe_destroy(None) == 0
    # quantiser: K not a multiple of 16, misaligned pointers, empty sizes
    assert lib.moe_quantize_nvfp4(0x1000, 1, 4, 24, 0x2000, 0x3000, 0x4000, None) == 1
    assert lib.moe_quantize_nvfp4(0x1004, 1, 4, 32, 0x2000, 0x3000, 0x4000, None) == 1
    assert lib.moe_quantize_nvfp4(0x1000, 0, 4, 32, 0x2000, 0x3000, 0x4000, None) == 1
    assert lib.moe_kernels_per_forward(None, 1, 0) == 0
    assert lib.moe_dense_kernels_per_forward(None, 1) == 0
