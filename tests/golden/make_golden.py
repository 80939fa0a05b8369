"""Write tests/golden/tiny_layer_oracle.txt: the oracle's output on the tiny workload.

Calls only the oracle and the seeded input generators.  The file is a
regression guard for the oracle itself (the pages print no worked example):
d_model 256, 16 routed experts top-2 + 1 shared, d_ff 128, bf16 weights
~N(0, 0.02), fp32 router ~N(0, 0.02), 4 bf16 tokens ~N(0, 1), seed 0.

    python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import synth  # noqa: E402
from oracle import moe  # noqa: E402


def tiny_layer_bf16(seed=0):
    s = synth.TINY
    wg, wu, wd = synth.expert_weights(s, seed)
    router = synth.router_weight(s, seed)
    bf = lambda t: t.to(torch.bfloat16).double().numpy()  # noqa: E731
    lw = moe.LayerWeights(router=router.numpy(), bias=None,
                          dense_gate=bf(wg), dense_up=bf(wu), dense_down=bf(wd))
    _, x = synth.tokens(s, 4, seed)
    return lw, x.double().numpy()


def main():
    lw, x = tiny_layer_bf16()
    r = moe.moe_layer(lw, x, k=synth.TINY.top_k, n_shared=synth.TINY.n_shared)
    out = os.path.join(HERE, "tiny_layer_oracle.txt")
    with open(out, "w") as fh:
        fh.write("# oracle output, tiny bf16-weight layer, seed 0 (written by make_golden.py)\n")
        fh.write("idx " + " ".join(str(int(v)) for v in r.idx.ravel()) + "\n")
        fh.write("w " + " ".join(repr(float(v)) for v in r.w.ravel()) + "\n")
        fh.write("y_bf16 " + " ".join(repr(float(v)) for v in r.y_bf16.ravel()) + "\n")
    print("wrote", out)


if __name__ == "__main__":
    main()
