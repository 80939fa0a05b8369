"""Build (nvcc, sm_103a) and run the microbenchmarks of this directory on GPU 0.

    python nvfp4_expert_ffn_gemv_b300/microbench/run.py [name ...]

Names: sync_burst_reduce, handoff, burst_issue, reduce_patterns, tma_stream, mma_rate,
tmem_a_mma, mxf4_n256, splitf_tail
(default: all).  Each prints its measurements; the summaries under profiles/
quote them.  Binaries go to _build/microbench/.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
OUT = os.path.join(os.path.dirname(os.path.dirname(HERE)), "_build", "microbench")
NAMES = ("sync_burst_reduce", "handoff", "burst_issue", "reduce_patterns", "tma_stream", "mma_rate", "tmem_a_mma",
         "mxf4_n256", "splitf_tail")


def main(names):
    os.makedirs(OUT, exist_ok=True)
    rc = 0
    for n in names:
        exe = os.path.join(OUT, n)
        subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-o", exe,
                        os.path.join(HERE, n + ".cu")], check=True)
        print(f"== {n}", flush=True)
        rc |= subprocess.run([exe]).returncode
    return rc


if __name__ == "__main__":
    sys.exit(main(sys.argv[1:] or NAMES))
