"""Writes tiny_t4_h256_shifted.txt: the CPU oracle's outputs for the tiny
shifted workload (4 tokens x hidden 256, seed 0), as exact bit patterns.
Calls only the oracle and the seeded input generator. Rerun it only when a
change to the oracle's arithmetic is intended, and name the passage that
justifies the change in the commit that updates the file.

    python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle as orc  # noqa: E402
from manifold_constrained_hyper_gb300 import synth  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_t4_h256_shifted.txt")


def oracle_outputs() -> dict:
    d = synth.workload_inputs("tiny_t4_h256")
    o = orc.boundary(orc.MODE_FUSED_SHIFTED, d["residual"], d["fn"], d["scale"], d["base"],
                     d["norm_w"], x=d["x"], post_mix=d["post"], comb=d["comb"],
                     pre_lag=d["pre_lag"])
    return {k: o[k] for k in ("residual_out", "layer_input", "pre", "post", "comb", "rstd",
                              "rstd_li")}


def encode(name: str, a: np.ndarray) -> str:
    bits = a.view(np.uint16 if a.dtype == np.uint16 else np.uint32).reshape(-1)
    width = 4 if a.dtype == np.uint16 else 8
    return f"{name} {a.dtype} {' '.join(str(s) for s in a.shape)}\n" + " ".join(
        f"{int(b):0{width}x}" for b in bits) + "\n"


def main():
    with open(OUT, "w") as f:
        f.write("# CPU oracle, tiny shifted workload (T=4, H=256, seed 0); bit patterns in hex\n")
        for k, v in oracle_outputs().items():
            f.write(encode(k, np.ascontiguousarray(v)))
    print("wrote", OUT)


if __name__ == "__main__":
    main()
