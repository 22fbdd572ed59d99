"""ctypes declarations of libmoe.so (include/moe.h).  Marshalling only."""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_CUDA = 3
MOE_ERR_TIMEOUT = 4
MOE_ERR_NONFINITE = 5

MOE_HAS_SHARED = 1
MOE_HAS_SHARED_GATE = 2
MOE_NO_FUSED = 4
MOE_PDL = 8
MOE_TENSOR_CORES = 16

# every symbol include/moe.h declares
EXPORTS = (
    "moe_packed_expert_bytes",
    "moe_workspace_bytes",
    "moe_workspace_init",
    "moe_pack_weights",
    "moe_route",
    "moe_expert_forward",
    "moe_layer_decode",
    "moe_stack_decode",
    "moe_layer_decode_noalloc",
    "moe_noalloc_test_timeout_next",
    "moe_get_device_status",
    "moe_status_string",
    "moe_last_error_message",
)


class moe_dims(ctypes.Structure):
    _fields_ = [
        ("hidden", ctypes.c_int32),
        ("inter", ctypes.c_int32),
        ("n_experts", ctypes.c_int32),
        ("top_k", ctypes.c_int32),
        ("bits", ctypes.c_int32),
        ("group", ctypes.c_int32),
        ("rms_eps", ctypes.c_float),
        ("flags", ctypes.c_int32),
    ]


class moe_layer(ctypes.Structure):
    _fields_ = [
        ("d", moe_dims),
        ("experts", ctypes.c_void_p),
        ("expert_stride", ctypes.c_size_t),
        ("shared", ctypes.c_void_p),
        ("shared_bits", ctypes.c_int32),
        ("router", ctypes.c_void_p),
        ("rms_gamma", ctypes.c_void_p),
        ("shared_gate", ctypes.c_void_p),
    ]


_lib = None


def load() -> ctypes.CDLL:
    """Load libmoe.so; raise loudly when it is missing (there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} not found: the CUDA library must be built (python -m bit_expert_matvec_moe_b300.build)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, SZ, VP = ctypes.POINTER, ctypes.c_int32, ctypes.c_size_t, ctypes.c_void_p
    lib.moe_packed_expert_bytes.restype = SZ
    lib.moe_packed_expert_bytes.argtypes = [P(moe_dims), I32]
    lib.moe_workspace_bytes.restype = SZ
    lib.moe_workspace_bytes.argtypes = [P(moe_dims), I32]
    lib.moe_workspace_init.restype = ctypes.c_int
    lib.moe_workspace_init.argtypes = [VP, SZ, VP]
    lib.moe_pack_weights.restype = ctypes.c_int
    lib.moe_pack_weights.argtypes = [P(moe_dims), I32, VP * 3, VP * 3, VP * 3, VP, VP]
    lib.moe_route.restype = ctypes.c_int
    lib.moe_route.argtypes = [P(moe_dims), VP, I32, VP, VP, VP, VP, VP, VP, SZ, VP]
    lib.moe_expert_forward.restype = ctypes.c_int
    lib.moe_expert_forward.argtypes = [P(moe_dims), I32, VP, VP, I32, VP, VP, I32, VP, SZ, VP]
    lib.moe_layer_decode.restype = ctypes.c_int
    lib.moe_layer_decode.argtypes = [P(moe_layer), VP, I32, VP, VP, VP, VP, SZ, VP]
    lib.moe_stack_decode.restype = ctypes.c_int
    lib.moe_stack_decode.argtypes = [P(moe_layer), I32, VP, VP, VP, VP, VP, SZ, VP]
    lib.moe_layer_decode_noalloc.restype = ctypes.c_int
    lib.moe_layer_decode_noalloc.argtypes = [P(moe_layer), VP, VP, VP, VP, VP, VP]
    lib.moe_noalloc_test_timeout_next.restype = ctypes.c_int
    lib.moe_noalloc_test_timeout_next.argtypes = []
    lib.moe_get_device_status.restype = ctypes.c_int
    lib.moe_get_device_status.argtypes = [VP, VP]
    lib.moe_status_string.restype = ctypes.c_char_p
    lib.moe_status_string.argtypes = [ctypes.c_int]
    lib.moe_last_error_message.restype = ctypes.c_char_p
    lib.moe_last_error_message.argtypes = []
    _lib = lib
    return lib
