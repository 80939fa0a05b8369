"""GPU parity at the edges of the shapes the library accepts.

* The widest routing: top_k = 8 with 2 shared experts, ten positions per
  token, the limit of every kernel that writes a token's positions (the
  batch-1 chain, bucketing, the batched-decode kernels, the prefill token
  quantiser and its scatter into the GEMM rows).
* The widest model: d_model = 4096 (the largest moe_init takes), through the
  same three paths.

Each shape runs batch 1, a ragged batch and a 64-token batch through decode,
and prefill batches whose shared experts span several 128-row blocks, against
the C++ oracle with the checks of the decode and prefill suites (routing and
combine weights within the fp32 logit bound, bf16 outputs within the
relative-L2 / max-abs bar, prefill h codes exact away from rounding midpoints).
"""
import pytest
import torch

import synth
from tests import harness
from tests.test_gpu_decode import check_layer
from tests.test_gpu_prefill import check_prefill

pytestmark = pytest.mark.gpu

WIDE_ROUTING = synth.MoEShape(d_model=256, n_experts=32, top_k=8, d_ff=256, n_shared=2)
WIDE_MODEL = synth.MoEShape(d_model=4096, n_experts=16, top_k=2, d_ff=256, n_shared=1)


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import nvfp4_expert_ffn_gemv_b300 as lib
    return lib


@pytest.mark.parametrize("shape", [WIDE_ROUTING, WIDE_MODEL], ids=["top8_shared2", "d4096"])
def test_edge_shape_decode_and_prefill(lib, shape):
    layer = harness.make_layer(lib, shape, seed=31, router_seed=32, fmt=0, max_tokens=512)
    try:
        for T in (1, 5, 64):
            xb, x = synth.tokens(shape, T, seed=900 + T)
            check_layer(lib, layer, xb.cuda(), x.numpy(), T,
                        prefix=f"d_model={shape.d_model} top_k={shape.top_k} S={shape.n_shared}")
        for T in (37, 300):
            xb, x = synth.tokens(shape, T, seed=950 + T)
            check_prefill(lib, layer, xb.cuda(), x.numpy(), T)
    finally:
        lib.moe_destroy(layer.ctx)
