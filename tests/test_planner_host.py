"""The decode matvec planner's invariants (shared memory within a CTA's limit,
2..8 stages, chunks covering each row exactly, row segments large enough for a
chunk's aligned superset, staged activations sized by their formula, a
multi-chunk row group no wider than the decode width) over a sweep of formats
and shapes, by a host-only program built with nvcc.  No GPU is touched."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_planner_invariants(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    exe = str(tmp_path / "planner_check")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17", "--expt-relaxed-constexpr",
                    "-I" + os.path.join(ROOT, "include"),
                    "-I" + os.path.join(ROOT, "gguf_block_quantised_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "planner_check.cu"), "-o", exe, "-lcudart"],
                   check=True, capture_output=True, text=True, timeout=600)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout[-3000:]
    assert "violations 0" in r.stdout
