"""Host-side checks of the kernels' work split (work_split.cuh), compiled
with nvcc as a plain host program: the equal split of numbered steps over
CTAs and its inverse, the prefill request step counts, and the split of
the SMs between the prefill tiles and the decode rows of a mixed batch.
No GPU is needed."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else shutil.which("nvcc")


def test_work_split_host_checks(tmp_path):
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not available")
    exe = str(tmp_path / "work_split_check")
    src = os.path.join(HERE, "host", "work_split_check.cu")
    build = subprocess.run(
        [nvcc, "-std=c++17", "-O1", "-gencode", "arch=compute_103a,code=sm_103a",
         "-I", os.path.join(ROOT, "include"),
         "-I", os.path.join(ROOT, "paged_kv_cache_74_gb300", "csrc"), src, "-o", exe],
        capture_output=True, text=True)
    assert build.returncode == 0, build.stderr
    run = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0 and run.stdout.strip() == "ok", run.stdout + run.stderr
