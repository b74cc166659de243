"""The performance diagnostics build for sm_103a without a GPU: the standalone MMA
issue-rate probe (csrc/issue_probe.cu) cross-compiles with nvcc."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "polynomial_matrix_whitening_gb300", "csrc")


@pytest.mark.skipif(shutil.which("nvcc") is None, reason="nvcc not installed")
def test_issue_probe_compiles(tmp_path):
    subprocess.check_call(["nvcc", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a",
                           "-I", CSRC, "-I", os.path.join(ROOT, "include"), "-c",
                           os.path.join(CSRC, "issue_probe.cu"), "-o", str(tmp_path / "issue_probe.o")])
    assert (tmp_path / "issue_probe.o").stat().st_size > 0
