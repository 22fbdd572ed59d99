"""Shared-memory plans and tile geometry, checked on the host with small
harnesses compiled by nvcc against the kernel files (no GPU needed):
tests/plan_check.cu checks the single-token kernel's plan for the shapes the
tests and the bench use and 3000 random shapes inside its limits (regions
aligned, disjoint and inside the total, per-block rows and copies inside their
slots, every row covered by the lane and thread mappings); tests/tile_check.cu
checks the batched path's tiles for every hidden and inter size the ABI
accepts; tests/tc_check.cu checks the tensor-core contraction's unpacking
tables against the packed format, its descriptor encodings, swizzle and
shared-memory plan."""
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


def _build_and_run(tmp_path, name, sources):
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not available")
    exe = str(tmp_path / name)
    cmd = [nvcc, "-std=c++17", "-O1", "-gencode", "arch=compute_103a,code=sm_103a", "-I",
           os.path.join(ROOT, "include"), *sources, "-o", exe]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stdout + res.stderr
    run = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, run.stdout + run.stderr
    words = run.stdout.split()
    assert words[0] == "ok" and int(words[1]) > 0, run.stdout


def test_single_token_plan_invariants(tmp_path):
    _build_and_run(tmp_path, "plan_check", [os.path.join(ROOT, "tests", "plan_check.cu"),
                                            os.path.join(ROOT, "bit_expert_matvec_moe_b300", "csrc", "moe_decode_b1.cu")])


def test_batched_tile_geometry(tmp_path):
    _build_and_run(tmp_path, "tile_check", [os.path.join(ROOT, "tests", "tile_check.cu")])


def test_tensor_core_tables_and_descriptors(tmp_path):
    _build_and_run(tmp_path, "tc_check", [os.path.join(ROOT, "tests", "tc_check.cu")])
