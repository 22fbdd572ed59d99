"""The single-token kernel's shared-memory plan, checked on the host: a small
harness (tests/plan_check.cu) is compiled with nvcc against the kernel file and
run; it checks the shapes the tests and the bench use and 3000 random shapes
inside the kernel's limits (regions aligned, disjoint and inside the total,
per-block rows and copies inside their slots, every row covered by the lane
and thread mappings).  No GPU needed."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    return None


def test_single_token_plan_invariants(tmp_path):
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not available")
    exe = str(tmp_path / "plan_check")
    cmd = [nvcc, "-std=c++17", "-O1", "-gencode", "arch=compute_103a,code=sm_103a", "-I",
           os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "plan_check.cu"),
           os.path.join(ROOT, "bit_expert_matvec_moe_b300", "csrc", "moe_decode_b1.cu"), "-o", exe]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stdout + res.stderr
    run = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, run.stdout + run.stderr
    words = run.stdout.split()
    assert words[0] == "ok" and int(words[1]) > 0, run.stdout
