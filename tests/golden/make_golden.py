"""Writes tests/golden/tiny_oracle.txt from the FP64 oracle alone.

Run: python tests/golden/make_golden.py
The file pins the oracle's output on the tiny workload (T=1, H=256, 8 routed
+ 1 shared experts, top-2, I=128, seed 0) against accidental changes; the
values come only from oracle/, never from the CUDA library.
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from block_scaled_fp4_moe_gb300 import inputs  # noqa: E402


def compute():
    cfg = inputs.CONFIGS["tiny"]
    x = inputs.make_x(cfg)
    wr, bias = inputs.make_router(cfg)
    bank = inputs.make_bank(cfg)
    return oracle.layer_forward(x, wr, bias, cfg.top_k, lambda e: {k: v[e] for k, v in bank.items()})


def main():
    out = compute()
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle.txt")
    with open(path, "w") as f:
        f.write("# FP64 oracle on the tiny workload (seed 0); written by make_golden.py\n")
        f.write("ids " + " ".join(str(int(v)) for v in out["ids"].ravel()) + "\n")
        f.write("w " + " ".join(repr(float(v)) for v in out["w"].ravel()) + "\n")
        f.write("y_bf16 " + " ".join("%04x" % int(v) for v in out["y_bf16"].ravel()) + "\n")
        f.write("y " + " ".join(repr(float(v)) for v in out["y"].ravel()) + "\n")


if __name__ == "__main__":
    main()
