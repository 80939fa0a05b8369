"""CPU oracle for the NVFP4 sparse-MoE FFN layer -- TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct numpy implementation (fp64 arithmetic unless
a step's precision is part of its definition) of what the CUDA library
computes.  It exists to check that library and shares no code with it: it
imports nothing from ``nvfp4_expert_ffn_gemv_b300`` and the library imports
nothing from here.  Only the test suite, the smoke check and the benchmark's
CPU-baseline / reference arm may import this package; the product path never
does and fails loudly instead of falling back to it.

Sources.  The method is the MoE FFN layer of Recursive Flint 40B-A2.5B as the
pages describe it:

* "Recursive Flint 40B-A2.5B：まず速さを第一に考えて作られたコーディングモデル"
  (OrcaRouter blog, ja), section "このアーキテクチャはメモリ帯域幅に関する主張である":
  256 routed experts per MoE layer, 6 chosen per token, one always-on shared
  expert, 47 of 49 layers are MoE; decode is a weight-bandwidth problem.
* same page, section "量子化のレシピは最も転用しやすい部分です": weights ship in
  NVFP4 (the format is named, not defined).
* "Recursive「Flint」とは。AIが作ったAIがノートPCで動く理由" (workwonders.jp),
  section "混合エキスパート（MoE）の仕組み": the same expert counts.

The pages print no formula, no layout and no worked example.  Every step they
leave open is taken in its plainest reading and listed where it is used:
softmax router with renormalised top-k, SwiGLU experts without biases,
d_model = 2048 and d_ff = 512, NVFP4 = E2M1 codes with one E4M3 scale per 16
elements along K and one FP32 scale per (expert, matrix), shared expert with
weight 1.

Pinning.  Every function here is checked by ``tests/test_oracle_*.py``
against something other than itself: torch's float8_e4m3fn conversions,
brute-force enumeration, closed-form bounds and invariants, and the page
figures under ``tests/golden/``.  Functions without such a pin say so.
"""
from . import nvfp4, moe  # noqa: F401
