"""Consistency pins from the figures the Flint pages print (tests/golden/flint_page_figures.txt).

The pages print no numerical example of the layer, so these pin the shapes
and the weight format, not outputs:

* BF16 checkpoint bytes ~= 2 bytes x 39.8B parameters;
* NVFP4 bytes ~= 4.5 bits x 39.8B parameters (E2M1 plus one 1-byte scale per
  16 elements), within 3% of the 22.86 GB file -- a 32-element block (4.25
  bits) lands 7.7% low and fails, as does a 2-byte scale;
* the routed + shared experts of 47 layers at d=2048, f=512 fit inside the
  39.8B total, and the active experts plus attention stay within the ~2.2B
  active body;
* "71% smaller" is 1 - 22.86 / 79.59;
* the readings of the two sizes the pages leave open -- the output layer's
  vocabulary (151,936 rows at d = 2048) and the dense layers' width (18,432)
  -- fit the counts: ~2.5B active with the head minus ~2.2B without it is the
  head, and what the 39.8B total and the ~2.2B active body leave after the
  experts, routers, attention and (untied) embedding and head is the two
  dense SwiGLU FFNs, each within the rounding of the printed figures.
"""
import os

import numpy as np

from oracle import nvfp4

HERE = os.path.dirname(os.path.abspath(__file__))


def _figures():
    out = {}
    with open(os.path.join(HERE, "golden", "flint_page_figures.txt"), encoding="utf-8") as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = (s.strip() for s in line.split("="))
                out[k] = float(v)
    return out


def _bits_per_weight(block: int, scale_bytes: int) -> float:
    """Storage of the oracle's NVFP4 layout for one [rows, K] tensor, per element."""
    rows, K = 512, 2048
    w = np.zeros((rows, K), np.float32)
    codes, scales, _ = nvfp4.quantize(w)
    assert codes.shape == (rows, K // 2) and scales.shape == (rows, K // 16)
    return 8 * (codes.nbytes + rows * (K // block) * scale_bytes) / (rows * K)


def test_checkpoint_sizes_support_16_element_e4m3_blocks():
    f = _figures()
    n = f["params_total_billion"] * 1e9
    assert abs(2 * n / 1e9 - f["bf16_checkpoint_gb"]) / f["bf16_checkpoint_gb"] < 0.01
    nvfp4_gb = n * _bits_per_weight(16, 1) / 8 / 1e9
    assert _bits_per_weight(16, 1) == 4.5
    assert abs(nvfp4_gb - f["nvfp4_gguf_gb"]) / f["nvfp4_gguf_gb"] < 0.03
    for block, sb in ((32, 1), (16, 2)):
        alt = n * (4 + 8 * sb / block) / 8 / 1e9
        assert abs(alt - f["nvfp4_gguf_gb"]) / f["nvfp4_gguf_gb"] > 0.05
    assert round(100 * (1 - f["nvfp4_gguf_gb"] / f["bf16_checkpoint_gb"])) == f["size_reduction_pct"]


def test_layer_shape_fits_parameter_budget():
    f = _figures()
    d, ff = 2048, 512
    per_expert = 3 * d * ff
    assert per_expert == 3_145_728
    n_moe = int(f["layers_moe"])
    assert int(f["layers_total"]) - n_moe == 2
    moe_total = n_moe * (f["routed_experts_per_layer"] + f["shared_experts"]) * per_expert
    assert moe_total < f["params_total_billion"] * 1e9
    active_moe = n_moe * (f["experts_per_token"] + f["shared_experts"]) * per_expert
    hd = f["head_dim"]
    attn = d * f["query_heads"] * hd * 2 + d * f["kv_heads"] * hd * 2
    active = active_moe + f["layers_total"] * attn
    assert active <= f["active_body_billion"] * 1e9 * 1.05
    # NVFP4 bytes of one expert: codes + one E4M3 byte per 16 elements
    assert per_expert // 2 + per_expert // 16 == 1_769_472


def test_head_and_dense_widths_fit_page_counts():
    import synth
    f = _figures()
    d = 2048
    head = synth.FLINT_VOCAB * d
    assert abs(head - (f["active_with_head_billion"] - f["active_body_billion"]) * 1e9) <= 0.1e9
    per_expert = 3 * d * 512
    n_moe = int(f["layers_moe"])
    n_dense = int(f["layers_total"]) - n_moe
    hd = f["head_dim"]
    attn = f["layers_total"] * (d * f["query_heads"] * hd * 2 + d * f["kv_heads"] * hd * 2)
    routers = n_moe * d * f["routed_experts_per_layer"]
    dense = n_dense * 3 * d * synth.FLINT_DENSE_FF
    left_total = (f["params_total_billion"] * 1e9
                  - n_moe * (f["routed_experts_per_layer"] + f["shared_experts"]) * per_expert
                  - routers - attn - 2 * head)
    left_active = (f["active_body_billion"] * 1e9
                   - n_moe * (f["experts_per_token"] + f["shared_experts"]) * per_expert - routers - attn)
    assert abs(dense - left_total) <= 0.05e9, (dense, left_total)
    assert abs(dense - left_active) <= 0.05e9, (dense, left_active)
