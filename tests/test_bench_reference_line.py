"""The reference arm of bench.py (the fp64 oracle on the host cores) prints one
JSON line with the keys the benchmark contract asks for; it needs no GPU."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "0", "--cpu-seconds", "1"], capture_output=True, text=True, timeout=600,
                         cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, res.stdout
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert "workload" in d["config"]


def test_profile_hash_ignores_comments_only():
    """A committed ncu capture stays valid while the kernel code hashes the
    same: rewording a comment keeps the hash, a change of code changes it."""
    import shutil
    import tempfile

    sys.path.insert(0, ROOT)
    import bench

    files = ("moe_decode_b1.cu", "moe_device.cuh", "moe_kernels.cu")
    with tempfile.TemporaryDirectory() as tmp:
        src = os.path.join(ROOT, "bit_expert_matvec_moe_b300", "csrc")
        dst = os.path.join(tmp, "bit_expert_matvec_moe_b300", "csrc")
        shutil.copytree(src, dst)
        base = bench.kernel_source_sha(files, root=tmp)
        path = os.path.join(dst, "moe_decode_b1.cu")
        text = open(path, encoding="utf-8").read()
        open(path, "w", encoding="utf-8").write("// another wording\n/* a block\n   comment */\n" + text + "\n  // tail\n")
        assert bench.kernel_source_sha(files, root=tmp) == base
        open(path, "w", encoding="utf-8").write(text.replace("kBlock - 32", "kBlock - 64", 1))
        assert bench.kernel_source_sha(files, root=tmp) != base
