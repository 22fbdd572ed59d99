"""C-ABI checks that need no GPU: the library loads, exports every function the
header declares, sizes are right, and host-side validation rejects bad
arguments before anything is enqueued."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def lib():
    from bit_expert_matvec_moe_b300 import build

    build.build()
    from bit_expert_matvec_moe_b300 import _native

    return _native.load()


def header_functions():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", txt)))


def test_exports_match_header(lib):
    from bit_expert_matvec_moe_b300 import _native

    declared = header_functions()
    assert declared == sorted(_native.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name  # dlsym succeeds


def dims(**kw):
    from bit_expert_matvec_moe_b300 import _native as N

    base = dict(hidden=4096, inter=1024, n_experts=512, top_k=4, bits=4, group=64, rms_eps=1e-6, flags=1)
    base.update(kw)
    return N.moe_dims(**base)


def test_packed_sizes(lib):
    d = dims()
    assert lib.moe_packed_expert_bytes(ctypes.byref(d), 4) == 7_077_888  # the pages' 6.75 MB
    assert lib.moe_packed_expert_bytes(ctypes.byref(d), 2) == 3_932_160
    t = dims(hidden=256, inter=128, n_experts=16)
    # tiny rows are padded to 16 bytes: down rows 64 + 8 -> 80 bytes
    assert lib.moe_packed_expert_bytes(ctypes.byref(t), 4) == 128 * 288 + 256 * 80
    assert lib.moe_packed_expert_bytes(ctypes.byref(t), 3) == 0


@pytest.mark.parametrize("bad", [
    dict(group=32), dict(hidden=100), dict(inter=0), dict(top_k=0), dict(top_k=9), dict(n_experts=2, top_k=3),
    dict(bits=3), dict(rms_eps=-1.0), dict(flags=2), dict(flags=64), dict(n_experts=2000),
])
def test_invalid_dims_rejected(lib, bad):
    d = dims(**bad)
    assert lib.moe_packed_expert_bytes(ctypes.byref(d), 4) == 0
    assert lib.moe_workspace_bytes(ctypes.byref(d), 1) == 0


def test_workspace_bytes_grows_with_batch(lib):
    d = dims()
    w1 = lib.moe_workspace_bytes(ctypes.byref(d), 1)
    w8 = lib.moe_workspace_bytes(ctypes.byref(d), 8)
    assert 0 < w1 < w8
    assert lib.moe_workspace_bytes(ctypes.byref(d), 0) == 0
    assert lib.moe_workspace_bytes(ctypes.byref(d), 257) == 0


def test_host_validation_returns_before_launch(lib):
    from bit_expert_matvec_moe_b300 import _native as N

    d = dims()
    VP3 = ctypes.c_void_p * 3
    # NULL / misaligned pointers: rejected on the host, no CUDA call made
    assert lib.moe_pack_weights(ctypes.byref(d), 4, VP3(None, None, None), VP3(None, None, None),
                                VP3(None, None, None), None, None) == N.MOE_ERR_INVALID_ARG
    assert lib.moe_route(ctypes.byref(d), None, 1, None, None, None, None, None, None, 0, None) == N.MOE_ERR_INVALID_ARG
    assert lib.moe_route(ctypes.byref(d), 16, 1, 32, None, 48, 64, None, 80, 10, None) == N.MOE_ERR_INVALID_ARG  # ws too small
    assert lib.moe_route(ctypes.byref(d), 17, 1, 32, None, 48, 64, None, 80, 1 << 30, None) == N.MOE_ERR_INVALID_ARG
    assert lib.moe_expert_forward(ctypes.byref(d), 4, None, None, 1, None, None, 0, None, 0, None) == N.MOE_ERR_INVALID_ARG
    assert lib.moe_expert_forward(ctypes.byref(d), 4, 16, 32, 0, None, 48, 0, 64, 1 << 30, None) == N.MOE_ERR_INVALID_ARG
    layer = N.moe_layer(d, None, 7_077_888, None, 4, None, None, None)
    assert lib.moe_layer_decode(ctypes.byref(layer), 16, 1, None, None, None, 32, 1 << 30, None) == N.MOE_ERR_INVALID_ARG
    layer = N.moe_layer(d, 16, 7_077_880, 32, 4, 48, None, None)  # stride below the blob size
    assert lib.moe_layer_decode(ctypes.byref(layer), 16, 1, None, None, None, 64, 1 << 30, None) == N.MOE_ERR_INVALID_ARG
    layer = N.moe_layer(d, 16, 7_077_888, 32, 3, 48, None, None)  # shared width 3
    assert lib.moe_layer_decode(ctypes.byref(layer), 16, 1, None, None, None, 64, 1 << 30, None) == N.MOE_ERR_INVALID_ARG
    layer = N.moe_layer(d, 16, 7_077_888, 32, 4, 48, None, None)
    assert lib.moe_layer_decode(ctypes.byref(layer), 16, 0, None, None, None, 64, 1 << 30, None) == N.MOE_ERR_INVALID_ARG
    assert lib.moe_layer_decode(ctypes.byref(layer), 16, 300, None, None, None, 64, 1 << 30, None) == N.MOE_ERR_INVALID_ARG
    assert lib.moe_get_device_status(None, None) == N.MOE_ERR_INVALID_ARG
    assert lib.moe_workspace_init(None, 0, None) == N.MOE_ERR_INVALID_ARG


def test_stack_decode_host_validation(lib):
    """moe_stack_decode refuses on the host (before any CUDA call): no layers,
    a null layer array, layers whose dims or shared widths differ, a bad layer
    among good ones, null or misaligned h, a small workspace."""
    from bit_expert_matvec_moe_b300 import _native as N

    d = dims()
    good = N.moe_layer(d, 16, 7_077_888, 32, 4, 48, None, None)
    ws = lib.moe_workspace_bytes(ctypes.byref(d), 1)
    arr = (N.moe_layer * 2)(good, good)
    assert lib.moe_stack_decode(arr, 0, 64, None, None, None, 80, ws, None) == N.MOE_ERR_INVALID_ARG
    assert lib.moe_stack_decode(None, 2, 64, None, None, None, 80, ws, None) == N.MOE_ERR_INVALID_ARG
    assert lib.moe_stack_decode(arr, 2, None, None, None, None, 80, ws, None) == N.MOE_ERR_INVALID_ARG
    assert lib.moe_stack_decode(arr, 2, 68, None, None, None, 80, ws, None) == N.MOE_ERR_INVALID_ARG
    assert lib.moe_stack_decode(arr, 2, 64, None, None, None, 80, ws - 16, None) == N.MOE_ERR_INVALID_ARG
    assert lib.moe_stack_decode(arr, 2, 64, 66, None, None, 80, ws, None) == N.MOE_ERR_INVALID_ARG  # offsets not 4-aligned
    other = N.moe_layer(dims(top_k=2), 16, 7_077_888, 32, 4, 48, None, None)
    assert lib.moe_stack_decode((N.moe_layer * 2)(good, other), 2, 64, None, None, None, 80, ws, None) == \
        N.MOE_ERR_INVALID_ARG
    two_bit_shared = N.moe_layer(d, 16, 7_077_888, 32, 2, 48, None, None)
    assert lib.moe_stack_decode((N.moe_layer * 2)(good, two_bit_shared), 2, 64, None, None, None, 80, ws, None) == \
        N.MOE_ERR_INVALID_ARG
    bad = N.moe_layer(d, None, 7_077_888, 32, 4, 48, None, None)
    assert lib.moe_stack_decode((N.moe_layer * 2)(good, bad), 2, 64, None, None, None, 80, ws, None) == \
        N.MOE_ERR_INVALID_ARG


def test_tensor_core_flag_workspace(lib):
    """MOE_TENSOR_CORES is a valid flag: the workspace grows by the tensor-core
    path's operand buffers (B rows of xn and of the activations, fp16 hi and lo,
    per (token, slot) entry), and a call without its buffers is refused on the
    host before anything is enqueued."""
    from bit_expert_matvec_moe_b300 import _native as N

    d = dims()
    t = dims(flags=1 | N.MOE_TENSOR_CORES)
    for B in (1, 8, 128):
        w0 = lib.moe_workspace_bytes(ctypes.byref(d), B)
        w1 = lib.moe_workspace_bytes(ctypes.byref(t), B)
        entries = B * (4 + 1)
        assert w1 - w0 >= entries * 2 * (4096 + 1024) * 2
    layer = N.moe_layer(t, 16, 7_077_888, 32, 4, 48, None, None)
    ws = lib.moe_workspace_bytes(ctypes.byref(t), 8)
    assert lib.moe_layer_decode(ctypes.byref(layer), None, 8, None, None, None, 64, ws, None) == N.MOE_ERR_INVALID_ARG
    assert lib.moe_layer_decode(ctypes.byref(layer), 16, 8, None, None, None, None, ws, None) == N.MOE_ERR_INVALID_ARG
    assert lib.moe_expert_forward(ctypes.byref(t), 4, None, 32, 3, None, 48, 0, 64, ws, None) == N.MOE_ERR_INVALID_ARG


def test_status_strings(lib):
    for s in range(6):
        assert lib.moe_status_string(s)
    assert lib.moe_status_string(99) == b"unknown status"


def test_product_path_does_not_import_oracle():
    """The package never imports the oracle or the input generator."""
    pkg = os.path.join(ROOT, "bit_expert_matvec_moe_b300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                txt = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in re.findall(r"import\s+(\w+)", txt)
                assert "from oracle" not in txt and "import oracle" not in txt
                assert "synth" not in re.findall(r"(?:from|import)\s+(\w+)", txt)
