"""The oracle still reproduces its committed output on the tiny workload (regression guard)."""
import os

import numpy as np

from oracle import moe
from tests.golden.make_golden import tiny_layer_bf16

HERE = os.path.dirname(os.path.abspath(__file__))


def test_tiny_layer_matches_committed_oracle_output():
    rows = {}
    with open(os.path.join(HERE, "golden", "tiny_layer_oracle.txt")) as fh:
        for line in fh:
            if not line.startswith("#"):
                key, *vals = line.split()
                rows[key] = np.array([float(v) for v in vals])
    lw, x = tiny_layer_bf16()
    r = moe.moe_layer(lw, x, k=2, n_shared=1)
    assert np.array_equal(r.idx.ravel(), rows["idx"].astype(np.int32))
    assert np.array_equal(r.w.ravel(), rows["w"])
    assert np.array_equal(r.y_bf16.ravel(), rows["y_bf16"])
