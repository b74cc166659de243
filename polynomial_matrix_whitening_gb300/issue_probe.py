"""How fast one thread can keep the 2-SM tensor pipe busy (csrc/issue_probe.cu).

Builds the standalone probe with nvcc (for sm_103a, into _build_probe/) and runs it on
the current GPU; prints a Markdown table of SM cycles per 64-deep k-block of 256 x 256
tiles for: the bare MMA chain, the chain with N dependent adds per k-block on the issuing
thread, and a 5-stage TMA ring whose issuer either waits for each stage's barrier or tests
the next stage's barrier while the current k-block's MMAs run (the cascade kernel's form).

  python -m polynomial_matrix_whitening_gb300.issue_probe
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def build() -> str:
    out_dir = os.path.join(HERE, "_build_probe")
    os.makedirs(out_dir, exist_ok=True)
    exe = os.path.join(out_dir, "issue_probe")
    src = os.path.join(HERE, "csrc", "issue_probe.cu")
    subprocess.check_call(["nvcc", "-O3", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a",
                           "-I", os.path.join(HERE, "csrc"), "-I", os.path.join(ROOT, "include"),
                           "-o", exe, src])
    return exe


def main() -> int:
    exe = build()
    return subprocess.call([exe])


if __name__ == "__main__":
    sys.exit(main())
