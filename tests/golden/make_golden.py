"""Writes tests/golden/tiny_layer_*.txt from the loop-only oracle (oracle.brute).

The stored values come only from ``oracle/``; rerun this script after a change
to the oracle's arithmetic that a cited passage justifies.

Workload: one fp32 layer, B=1, T=6, M=2 meta rows, d=8, 2 query heads and
1 KV head of dim 4 (dv = 4), di=8, N=2, k=4, window 3, RoPE base 10000,
inputs from the seeded generator (seed 11).  Definition followed: "Hymba: A
Hybrid-head Architecture for Small Language Models", section 2.1 eq. (3),
sections 2.2 and 2.3.
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from hybrid_attention_ssm_fwd_b300 import synth  # noqa: E402
from oracle import brute  # noqa: E402


def golden_shape(**kw):
    base = dict(B=1, T=6, M=2, d=8, Hq=2, Hkv=1, dh=4, di=8, N=2, k=4, window=3,
                rope_theta=10000.0)
    base.update(kw)
    return synth.tiny_f32(**base)


CASES = {"swa_rope": dict(), "global": dict(window=0, rope_theta=0.0)}


def main():
    for name, kw in CASES.items():
        s = golden_shape(**kw)
        p = synth.make_layer_inputs(s, 11)
        y = np.array(brute.layer_fwd(p, p["Xt"], s)["Y"])[0]
        path = os.path.join(HERE, f"tiny_layer_{name}.txt")
        with open(path, "w") as f:
            f.write(f"# Y[L={s.L}][d={s.d}] from oracle.brute, case {name}, seed 11\n")
            for row in y:
                f.write(" ".join(repr(float(v)) for v in row) + "\n")


if __name__ == "__main__":
    main()
