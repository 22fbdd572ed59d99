"""B300 (sm_103a) decode-time MoE expert path behind a C ABI (libmoe.so).

The functions here carry the names of the C entry points and only marshal
arguments: torch tensors supply device memory and the current CUDA stream,
every step of the path runs in the library's kernels.  There is no fallback:
importing works without a GPU, but each call needs the built library and a
CUDA device, and fails loudly otherwise.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

from . import _native as N
from ._native import MOE_HAS_SHARED, MOE_HAS_SHARED_GATE, MOE_NO_FUSED, MOE_PDL  # noqa: F401

__all__ = [
    "Dims", "MoeError", "moe_packed_expert_bytes", "moe_workspace_bytes", "moe_workspace_init",
    "moe_pack_weights", "moe_route", "moe_expert_forward", "moe_layer_decode", "moe_layer_decode_noalloc",
    "moe_get_device_status",
    "make_layer",
]


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = N.load()
        msg = lib.moe_status_string(status).decode()
        if status == N.MOE_ERR_CUDA:
            msg += ": " + lib.moe_last_error_message().decode()
        super().__init__(f"{where}: {msg}")
        self.status = status


@dataclass
class Dims:
    hidden: int
    inter: int
    n_experts: int
    top_k: int
    bits: int = 4
    group: int = 64
    rms_eps: float = 1e-6
    flags: int = MOE_HAS_SHARED

    def c(self) -> N.moe_dims:
        return N.moe_dims(self.hidden, self.inter, self.n_experts, self.top_k, self.bits, self.group,
                          self.rms_eps, self.flags)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream=None) -> int:
    import torch

    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check(rc: int, where: str) -> None:
    if rc != N.MOE_OK:
        raise MoeError(rc, where)


def moe_packed_expert_bytes(dims: Dims, bits: int) -> int:
    return int(N.load().moe_packed_expert_bytes(ctypes.byref(dims.c()), bits))


def moe_workspace_bytes(dims: Dims, max_batch: int) -> int:
    return int(N.load().moe_workspace_bytes(ctypes.byref(dims.c()), max_batch))


def moe_workspace_init(ws, stream=None) -> None:
    _check(N.load().moe_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)), "moe_workspace_init")


def moe_pack_weights(dims: Dims, bits: int, codes, scales, biases, dst, stream=None) -> None:
    """codes/scales/biases: three tensors each (gate, up, down), canonical layout."""
    VP3 = ctypes.c_void_p * 3
    c = VP3(*[_ptr(t) for t in codes])
    s = VP3(*[_ptr(t) for t in scales])
    b = VP3(*[_ptr(t) for t in biases])
    _check(N.load().moe_pack_weights(ctypes.byref(dims.c()), bits, c, s, b, _ptr(dst), _stream(stream)),
           "moe_pack_weights")


def moe_route(dims: Dims, xn, router, idx, w, ws, logit_offset=None, logits_out=None, stream=None) -> None:
    B = xn.shape[0]
    _check(N.load().moe_route(ctypes.byref(dims.c()), _ptr(xn), B, _ptr(router), _ptr(logit_offset), _ptr(idx),
                              _ptr(w), _ptr(logits_out), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "moe_route")


def moe_expert_forward(dims: Dims, bits: int, blob, xn, out, ws, row_w=None, accumulate: bool = False,
                       stream=None) -> None:
    B = xn.shape[0]
    _check(N.load().moe_expert_forward(ctypes.byref(dims.c()), bits, _ptr(blob), _ptr(xn), B, _ptr(row_w), _ptr(out),
                                       1 if accumulate else 0, _ptr(ws), ws.numel() * ws.element_size(),
                                       _stream(stream)),
           "moe_expert_forward")


def make_layer(dims: Dims, experts, expert_stride: int, router, shared=None, shared_bits: int = 4, rms_gamma=None,
               shared_gate=None) -> N.moe_layer:
    """A C moe_layer that refers to the given device tensors (keep them alive)."""
    return N.moe_layer(dims.c(), _ptr(experts), expert_stride, _ptr(shared), shared_bits, _ptr(router),
                       _ptr(rms_gamma), _ptr(shared_gate))


def moe_layer_decode(layer: N.moe_layer, h, ws, logit_offset=None, idx_out=None, w_out=None, stream=None) -> None:
    B = h.shape[0]
    _check(N.load().moe_layer_decode(ctypes.byref(layer), _ptr(h), B, _ptr(logit_offset), _ptr(idx_out), _ptr(w_out),
                                     _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "moe_layer_decode")


def moe_layer_decode_noalloc(layer: N.moe_layer, h, logit_offset=None, idx_out=None, w_out=None, status_out=None,
                             stream=None) -> None:
    """Single-token layer without a caller workspace (the library's fixed
    device array instead; see include/moe.h).  h is [1, hidden]."""
    if h.shape[0] != 1:
        raise ValueError("moe_layer_decode_noalloc takes one token")
    _check(N.load().moe_layer_decode_noalloc(ctypes.byref(layer), _ptr(h), _ptr(logit_offset), _ptr(idx_out),
                                             _ptr(w_out), _ptr(status_out), _stream(stream)),
           "moe_layer_decode_noalloc")


def moe_get_device_status(ws, stream=None) -> int:
    """Synchronise, read and clear the workspace status word (0 = ok)."""
    return int(N.load().moe_get_device_status(_ptr(ws), _stream(stream)))
