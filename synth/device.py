"""Device-side generation of the same canonical weights as synth.generate (the
CUDA twin in synth/csrc/synth_gen.cu).  Used by the benchmark and the tests for
layers too large to generate on the host."""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess

import torch

from . import generate as G

HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(HERE, "libsynth.so")
SRC = os.path.join(HERE, "csrc", "synth_gen.cu")


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
           "-shared", "-o", LIB + ".tmp", SRC]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + res.stdout + res.stderr)
    os.replace(LIB + ".tmp", LIB)
    return LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise ImportError(f"{LIB} is missing: run __graft_entry__.build()")
        _lib = ctypes.CDLL(LIB)
        _lib.synth_matrix.restype = ctypes.c_int
        _lib.synth_matrix.argtypes = [ctypes.c_uint64] * 4 + [ctypes.c_int] * 4 + [ctypes.c_void_p] * 4
        _lib.synth_stream_key.restype = ctypes.c_uint64
        _lib.synth_stream_key.argtypes = [ctypes.POINTER(ctypes.c_uint64), ctypes.c_int]
    return _lib


def stream_key(*fields: int) -> int:
    arr = (ctypes.c_uint64 * len(fields))(*[int(f) & G.MASK64 for f in fields])
    return int(_load().synth_stream_key(arr, len(fields)))


def matrix(seed, layer, expert, tensor, rows, cols, bits, group=64, device="cuda"):
    """Canonical (codes, scales, biases) tensors on `device`, equal bit for bit to
    synth.generate.matrix."""
    lib = _load()
    codes = torch.empty((rows, cols * bits // 8), dtype=torch.uint8, device=device)
    sc = torch.empty((rows, cols // group), dtype=torch.int16, device=device)
    bi = torch.empty((rows, cols // group), dtype=torch.int16, device=device)
    rc = lib.synth_matrix(seed, layer, expert, tensor, rows, cols, bits, group, codes.data_ptr(), sc.data_ptr(),
                          bi.data_ptr(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    if rc != 0:
        raise RuntimeError(f"synth_matrix failed: CUDA error {rc}")
    return codes, sc, bi


def expert(seed, layer, e, hidden, inter, bits, group=64, device="cuda"):
    return {
        "bits": bits,
        "group": group,
        "gate": matrix(seed, layer, e, G.T_GATE, inter, hidden, bits, group, device),
        "up": matrix(seed, layer, e, G.T_UP, inter, hidden, bits, group, device),
        "down": matrix(seed, layer, e, G.T_DOWN, hidden, inter, bits, group, device),
    }
