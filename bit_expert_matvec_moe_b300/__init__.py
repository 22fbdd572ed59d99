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
from ._native import MOE_HAS_SHARED, MOE_HAS_SHARED_GATE, MOE_NO_FUSED, MOE_PDL, MOE_TENSOR_CORES  # noqa: F401

__all__ = [
    "Dims", "MoeError", "moe_packed_expert_bytes", "moe_workspace_bytes", "moe_workspace_init",
    "moe_pack_weights", "moe_route", "moe_expert_forward", "moe_layer_decode", "moe_stack_decode",
    "moe_layer_decode_noalloc",
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


# element types the C ABI expects, by argument kind (dtype names of torch)
_KINDS = {
    "f32": ("float32",),
    "i32": ("int32",),
    "b16": ("int16", "uint16", "bfloat16"),  # bf16 bit patterns
    "u8": ("uint8", "int8"),
}


def _check_type(t, name: str, kind: str | None = None, numel: int | None = None) -> None:
    """Element type (kind) and size (at least `numel` elements) of a tensor argument."""
    if t is None or isinstance(t, int):
        return
    if kind is not None:
        dt = str(t.dtype).replace("torch.", "")
        if dt not in _KINDS[kind]:
            raise ValueError(f"{name}: expected dtype {' or '.join(_KINDS[kind])}, got {dt}")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name}: expected at least {numel} elements, got {t.numel()}")


def _ptr(t, name: str = "tensor", kind: str | None = None, numel: int | None = None) -> int | None:
    """Device pointer of a contiguous CUDA tensor (an integer is taken as a
    pointer as it is), after the checks of _check_type."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    _check_type(t, name, kind, numel)
    if not t.is_cuda:
        raise ValueError(f"{name}: expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous tensor")
    return t.data_ptr()


def _ptrs(*specs) -> list:
    """Pointers of several arguments (tensor, name, kind, numel): every type
    and size is checked first, so the error names the argument that is wrong."""
    for spec in specs:
        _check_type(*spec)
    return [_ptr(*spec) for spec in specs]


def _rows(t, name: str, cols: int) -> int:
    """Rows of a [B, cols] tensor."""
    if t.dim() != 2 or t.shape[1] != cols:
        raise ValueError(f"{name}: expected shape [B, {cols}], got {list(t.shape)}")
    return int(t.shape[0])


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
    ptrs = _ptrs(*[(t, "codes", "u8", None) for t in codes], *[(t, "scales", "b16", None) for t in scales],
                 *[(t, "biases", "b16", None) for t in biases])
    c, s, b = VP3(*ptrs[0:3]), VP3(*ptrs[3:6]), VP3(*ptrs[6:9])
    _check(N.load().moe_pack_weights(ctypes.byref(dims.c()), bits, c, s, b, _ptr(dst), _stream(stream)),
           "moe_pack_weights")


def moe_route(dims: Dims, xn, router, idx, w, ws, logit_offset=None, logits_out=None, stream=None) -> None:
    B = _rows(xn, "xn", dims.hidden)
    E, K = dims.n_experts, dims.top_k
    px, pr, po, pi, pw, pl = _ptrs((xn, "xn", "f32", None), (router, "router", "b16", E * dims.hidden),
                                   (logit_offset, "logit_offset", "f32", B * E), (idx, "idx", "i32", B * K),
                                   (w, "w", "f32", B * K), (logits_out, "logits_out", "f32", B * E))
    _check(N.load().moe_route(ctypes.byref(dims.c()), px, B, pr, po, pi, pw, pl, _ptr(ws),
                              ws.numel() * ws.element_size(), _stream(stream)),
           "moe_route")


def moe_expert_forward(dims: Dims, bits: int, blob, xn, out, ws, row_w=None, accumulate: bool = False,
                       stream=None) -> None:
    B = _rows(xn, "xn", dims.hidden)
    px, prw, po = _ptrs((xn, "xn", "f32", None), (row_w, "row_w", "f32", B), (out, "out", "f32", B * dims.hidden))
    _check(N.load().moe_expert_forward(ctypes.byref(dims.c()), bits, _ptr(blob), px, B, prw, po,
                                       1 if accumulate else 0, _ptr(ws), ws.numel() * ws.element_size(),
                                       _stream(stream)),
           "moe_expert_forward")


def make_layer(dims: Dims, experts, expert_stride: int, router, shared=None, shared_bits: int = 4, rms_gamma=None,
               shared_gate=None) -> N.moe_layer:
    """A C moe_layer that refers to the given device tensors (keep them alive)."""
    H = dims.hidden
    pr, pg, ps = _ptrs((router, "router", "b16", dims.n_experts * H), (rms_gamma, "rms_gamma", "b16", H),
                       (shared_gate, "shared_gate", "b16", H))
    return N.moe_layer(dims.c(), _ptr(experts), expert_stride, _ptr(shared), shared_bits, pr, pg, ps)


def _layer_io(layer, h, logit_offset, idx_out, w_out):
    d = layer.d
    B = _rows(h, "h", d.hidden)
    return B, _ptrs((h, "h", "f32", None), (logit_offset, "logit_offset", "f32", B * d.n_experts),
                    (idx_out, "idx_out", "i32", B * d.top_k), (w_out, "w_out", "f32", B * d.top_k))


def moe_layer_decode(layer: N.moe_layer, h, ws, logit_offset=None, idx_out=None, w_out=None, stream=None) -> None:
    B, (ph, po, pi, pw) = _layer_io(layer, h, logit_offset, idx_out, w_out)
    _check(N.load().moe_layer_decode(ctypes.byref(layer), ph, B, po, pi, pw, _ptr(ws), ws.numel() * ws.element_size(),
                                     _stream(stream)),
           "moe_layer_decode")


def moe_stack_decode(layers, h, ws, logit_offset=None, idx_out=None, w_out=None, stream=None) -> None:
    """One token through the layers in order, in place on h ([1, hidden] or
    [hidden]).  layers: a sequence of moe_layer of equal dims; logit_offset
    [n_layers, n_experts], idx_out / w_out [n_layers, top_k] (or None)."""
    layers = list(layers)
    if not layers:
        raise ValueError("moe_stack_decode: no layers")
    d = layers[0].d
    n = len(layers)
    if h.numel() != d.hidden:
        raise ValueError(f"moe_stack_decode: h must hold one token ({d.hidden} values)")
    arr = (N.moe_layer * n)(*layers)
    ph, po, pi, pw = _ptrs((h, "h", "f32", d.hidden), (logit_offset, "logit_offset", "f32", n * d.n_experts),
                           (idx_out, "idx_out", "i32", n * d.top_k), (w_out, "w_out", "f32", n * d.top_k))
    _check(N.load().moe_stack_decode(arr, n, ph, po, pi, pw, _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "moe_stack_decode")


def moe_layer_decode_noalloc(layer: N.moe_layer, h, status_out, logit_offset=None, idx_out=None, w_out=None,
                             stream=None) -> None:
    """Single-token layer without a caller workspace (the library's fixed
    device array instead; see include/moe.h).  h is [1, hidden]; status_out is
    a device int32 that receives the call's device status (required: it is the
    only record of a device-side error)."""
    if status_out is None:
        raise ValueError("moe_layer_decode_noalloc: status_out is required")
    B, (ph, po, pi, pw) = _layer_io(layer, h, logit_offset, idx_out, w_out)
    if B != 1:
        raise ValueError("moe_layer_decode_noalloc takes one token")
    _check(N.load().moe_layer_decode_noalloc(ctypes.byref(layer), ph, po, pi, pw, _ptr(status_out, "status_out", "i32", 1),
                                             _stream(stream)),
           "moe_layer_decode_noalloc")


def moe_get_device_status(ws, stream=None) -> int:
    """Synchronise, read and clear the workspace status word (0 = ok)."""
    return int(N.load().moe_get_device_status(_ptr(ws), _stream(stream)))
