"""The bench's N > 1 host logic on CPU: two gloo ranks run the replica bookkeeping
(barrier, max over ranks, whole-job value) the way torch.distributed.run would launch
them on two GPUs, and the reference arm runs on rank 0 only."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import os, sys, json
sys.path.insert(0, os.environ["ROOT"])
import bench
world, rank, local = bench.dist_setup()
assert world == 2 and rank in (0, 1)
bench.barrier(world)
ms_local = 1.0 + rank            # rank 1 is the slow one
ms, value = bench.job_value(ms_local, 66, world)
with open(os.path.join(os.environ["OUT_DIR"], f"rank{rank}.json"), "w") as f:
    json.dump({"rank": rank, "ms": ms, "value": value}, f)
import torch.distributed as dist
dist.destroy_process_group()
"""


def test_replica_timing_is_max_over_ranks(tmp_path):
    script = tmp_path / "w.py"
    script.write_text(WORKER)
    env = dict(os.environ, ROOT=ROOT, CUDA_VISIBLE_DEVICES="", OUT_DIR=str(tmp_path))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", "29531", str(script)]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    import json
    lines = [json.load(open(tmp_path / f"rank{k}.json")) for k in range(2)]
    assert sorted(l["rank"] for l in lines) == [0, 1]
    for l in lines:
        assert l["ms"] == 2.0                      # the slowest rank's time
        assert abs(l["value"] - 66 * 2 / 0.002) < 1e-6


@pytest.mark.slow
def test_reference_arm_prints_on_rank_zero_only(tmp_path):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", "29533", "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "1", "--warmup", "3", "--reference-budget", "4"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    import json
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1 and lines[0]["impl"] == "reference"
    assert lines[0]["value"] > 0 and lines[0]["cpu_baseline"]["kind"] == "oracle"


@pytest.mark.parametrize("visible,local,want", [
    (None, 0, "0"), (None, 3, "3"), ("4,5", 1, "5"), ("GPU-aa, GPU-bb", 1, "GPU-bb"), ("", 2, "2"),
])
def test_clock_sampler_gets_each_ranks_physical_gpu(monkeypatch, visible, local, want):
    """The clocks recorded beside a rank's number are its own GPU's: the id CUDA_VISIBLE_DEVICES
    lists for its local rank (index or UUID, as nvidia-smi -i takes them)."""
    sys.path.insert(0, ROOT)
    import bench
    if visible is None:
        monkeypatch.delenv("CUDA_VISIBLE_DEVICES", raising=False)
    else:
        monkeypatch.setenv("CUDA_VISIBLE_DEVICES", visible)
    assert bench.physical_gpu(local) == want
