"""The warp rings' walk replayed on the host (CPU): tests/walk_replay.cu
includes the plan and walkers the kernels use and checks bounds, 16-byte
alignment, exact coverage of every rank's input and output, and that the
own-data prefetch walk matches the stage walk, on random calls."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_walk_replay(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    exe = str(tmp_path / "walk_replay")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17",
                    "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(ROOT, "ring_allreduce_virtual_gb300", "csrc"),
                    os.path.join(HERE, "walk_replay.cu"), "-o", exe], check=True)
    r = subprocess.run([exe, "3000"], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    assert r.stdout.startswith("ok")
