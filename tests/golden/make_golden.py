"""Write the stored expected outputs under tests/golden/ from the CPU oracle only.

    python tests/golden/make_golden.py

Each fixture is the oracle's bf16 result for one seeded workload from
workloads.py, written as hex bit patterns, one output row per line.  Nothing
here comes from the CUDA path.
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import workloads as wl  # noqa: E402

FIXTURES = [
    # smallest MoE router case: M=4, K=2048, N=256, no bias, seed 0
    ("router_smallest_seed0.txt", dict(M=4, N=256, K=2048, seed=0, bias=False)),
    # ragged tiny case with bias: K=2880 (not a multiple of 64), N=17
    ("ragged_M3_N17_K2880_bias_seed7.txt", dict(M=3, N=17, K=2880, seed=7, bias=True)),
]


def write(name, M, N, K, seed, bias):
    x, W, b = wl.make_inputs(M, N, K, seed, bias)
    out = oracle.linear_bf16(wl.bits(x), wl.bits(W), wl.bits(b))
    with open(os.path.join(HERE, name), "w") as f:
        f.write(f"# oracle bf16 out[M,N] hex, M={M} N={N} K={K} seed={seed} bias={int(bias)}\n")
        f.write("# inputs: workloads.make_inputs (x~N(0,1), W~N(0,1/K), bias~U(-0.1,0.1)), bf16\n")
        for row in out:
            f.write(" ".join(f"{int(v):04x}" for v in row) + "\n")


def read(name):
    import numpy as np
    rows = []
    meta = None
    with open(os.path.join(HERE, name)) as f:
        for line in f:
            if line.startswith("#"):
                if meta is None and "M=" in line:
                    meta = dict(kv.split("=") for kv in line.split() if "=" in kv)
                continue
            rows.append([int(t, 16) for t in line.split()])
    return {k: int(v) for k, v in meta.items()}, np.array(rows, dtype=np.uint16)


if __name__ == "__main__":
    for name, cfg in FIXTURES:
        write(name, **cfg)
        print("wrote", name)
