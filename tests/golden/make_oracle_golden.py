"""Writes tests/golden/oracle_small.txt: the oracle's output bits for three tiny seeded
cases (a regression fixture; it also shows that the oracle builds to the same bits on
x86-64 and aarch64).  Calls only oracle/ and the seeded input generators."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from polynomial_matrix_whitening_gb300 import workloads as W  # noqa: E402

CASES = [("wide", 1, 4, 6), ("tall", 1, 6, 4), ("square", 2, 5, 5)]


def compute():
    out = {}
    for name, g, m, n in CASES:
        grad, vel = W.random_case(100 + m * n, g, m, n)
        o, v = oracle.bank_step(grad, vel, 0.95, 0.85, 0.4385, 0.98)
        out[name] = (o, v)
    return out


def main():
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_small.txt")
    with open(path, "w") as f:
        f.write("# written by tests/golden/make_oracle_golden.py from oracle/ only\n")
        f.write("# case g m n: out bf16 bits (hex), then velocity fp32 bits (hex)\n")
        for (name, g, m, n), (o, v) in zip(CASES, compute().values()):
            f.write(f"case {name} {g} {m} {n}\n")
            f.write("out " + " ".join(f"{x:04x}" for x in o.ravel()) + "\n")
            f.write("vel " + " ".join(f"{x:08x}" for x in v.view("uint32").ravel()) + "\n")


if __name__ == "__main__":
    main()
