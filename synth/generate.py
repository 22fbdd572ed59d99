"""Seeded, counter-based synthetic inputs for the MoE decode path.

This module holds no arithmetic of the method itself: it only draws random
numbers and rounds them to storage types.  Both the fp64 oracle (through the
tests) and the CUDA path (through the benchmark and the tests) take their
inputs from here, so that the two sides see identical bytes.

Generator
---------
SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014; the 64-bit finaliser constants are Stafford's
"Mix13" variant as used by Vigna's public splitmix64.c).  A stream is named by
a tuple of integer fields; its key is

    k0 = 0x243F6A8885A308D3
    k_{n+1} = mix((k_n XOR field_n) + GAMMA)        (mod 2^64)

and its i-th 64-bit output (i = 0, 1, ...) is ``mix(key + (i + 1) * GAMMA)``,
which is exactly SplitMix64's (i+1)-th output when seeded with ``key``.
Because every output depends only on (key, i), any slice of any tensor can be
regenerated independently, on the host (this file) or on the device (the twin
in ``synth/csrc/synth_gen.cu``, which must produce the same bits).

Derived values
--------------
* uniform u in [0, 1):  (out >> 11) * 2^-53
* code bytes:           byte j of a tensor is byte (j mod 8) (little-endian)
                        of output j // 8; a uniform byte holds two uniform
                        4-bit codes or four uniform 2-bit codes
* scale  s:             bf16(f32(0.005 + 0.015 * u))            [fp64 ops]
* bias   b:             bf16(f32((-c * s) * (0.9 + 0.2 * u')))  c = 8 (4-bit), 1.5 (2-bit)
* normal z:             Box-Muller from outputs 2i, 2i+1 (host only)
Every fp64 step is a single correctly rounded IEEE operation (no fused
multiply-add), so the device twin reproduces it bit for bit.
"""
from __future__ import annotations

import numpy as np

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
KEY0 = 0x243F6A8885A308D3
SEED = 20260101

# Stream field values (tensor and part identifiers).
T_GATE, T_UP, T_DOWN, T_ROUTER, T_H, T_GAMMA, T_SHARED_GATE, T_OFFSET, T_TRACE = range(1, 10)
P_CODES, P_SCALES, P_BIASES, P_VALUES = range(1, 5)
SHARED_EXPERT = 0xFFFF  # expert field of the shared expert

_U64 = np.uint64


def _mix_int(z: int) -> int:
    z &= MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def stream_key(*fields: int) -> int:
    k = KEY0
    for f in fields:
        k = _mix_int(((k ^ (int(f) & MASK64)) + GAMMA) & MASK64)
    return k


def _mix_np(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = (z ^ (z >> _U64(30))) * _U64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> _U64(27))) * _U64(0x94D049BB133111EB)
        return z ^ (z >> _U64(31))


def raw64(key: int, start: int, count: int) -> np.ndarray:
    """Outputs start .. start+count-1 of the stream `key` (uint64)."""
    i = np.arange(start + 1, start + 1 + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = _U64(key) + i * _U64(GAMMA)
    return _mix_np(z)


def uniform(key: int, count: int, start: int = 0) -> np.ndarray:
    return (raw64(key, start, count) >> _U64(11)).astype(np.float64) * (2.0 ** -53)


def normal(key: int, count: int) -> np.ndarray:
    r = raw64(key, 0, 2 * count)
    u1 = ((r[0::2] >> _U64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)  # (0, 1]
    u2 = (r[1::2] >> _U64(11)).astype(np.float64) * (2.0 ** -53)
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


def code_bytes(key: int, nbytes: int) -> np.ndarray:
    n64 = (nbytes + 7) // 8
    return raw64(key, 0, n64).view(np.uint8)[:nbytes].copy()


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even float32 -> bfloat16 bit pattern (uint16); finite inputs."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + _U64(0x7FFF) + ((b >> _U64(16)) & _U64(1))) >> _U64(16)
    return b.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def scale_bias(seed: int, layer: int, expert: int, tensor: int, n: int, bits: int):
    """bf16 bit patterns of n scales and n biases for one weight matrix."""
    u = uniform(stream_key(seed, layer, expert, tensor, P_SCALES), n)
    s = 0.005 + 0.015 * u
    s_bf = f32_to_bf16_bits(s.astype(np.float32))
    s64 = bf16_bits_to_f32(s_bf).astype(np.float64)
    c = 8.0 if bits == 4 else 1.5
    v = 0.9 + 0.2 * uniform(stream_key(seed, layer, expert, tensor, P_BIASES), n)
    b = (-c * s64) * v
    return s_bf, f32_to_bf16_bits(b.astype(np.float32))


def matrix(seed: int, layer: int, expert: int, tensor: int, rows: int, cols: int,
           bits: int, group: int):
    """Canonical quantised matrix: codes uint8 [rows, cols*bits/8], scales and
    biases as bf16 bit patterns uint16 [rows, cols/group]."""
    nb = rows * cols * bits // 8
    codes = code_bytes(stream_key(seed, layer, expert, tensor, P_CODES), nb).reshape(rows, cols * bits // 8)
    s, b = scale_bias(seed, layer, expert, tensor, rows * (cols // group), bits)
    return codes, s.reshape(rows, cols // group), b.reshape(rows, cols // group)


def expert(seed: int, layer: int, e: int, hidden: int, inter: int, bits: int, group: int = 64):
    """One expert's three matrices: gate [I,H], up [I,H], down [H,I]."""
    return {
        "bits": bits,
        "group": group,
        "gate": matrix(seed, layer, e, T_GATE, inter, hidden, bits, group),
        "up": matrix(seed, layer, e, T_UP, inter, hidden, bits, group),
        "down": matrix(seed, layer, e, T_DOWN, hidden, inter, bits, group),
    }


def router(seed: int, layer: int, n_experts: int, hidden: int, std: float = 0.02) -> np.ndarray:
    z = normal(stream_key(seed, layer, 0, T_ROUTER, P_VALUES), n_experts * hidden)
    return f32_to_bf16_bits((std * z).astype(np.float32)).reshape(n_experts, hidden)


def hidden_states(seed: int, layer: int, tokens: int, hidden: int, stream: int = 0) -> np.ndarray:
    z = normal(stream_key(seed, layer, stream, T_H, P_VALUES), tokens * hidden)
    return z.astype(np.float32).reshape(tokens, hidden)


def bf16_vector(seed: int, layer: int, tensor: int, n: int, mean: float, std: float) -> np.ndarray:
    z = normal(stream_key(seed, layer, 0, tensor, P_VALUES), n)
    return f32_to_bf16_bits((mean + std * z).astype(np.float32))


def popularity_offsets(seed: int, layer: int, n_experts: int, std: float = 1.5) -> np.ndarray:
    """Per-expert logit offsets o_e ~ N(0, std) (skewed-routing workload)."""
    z = normal(stream_key(seed, layer, 0, T_OFFSET, P_VALUES), n_experts)
    return (std * z).astype(np.float32)


def reuse_trace(seed: int, layer: int, tokens: int, n_experts: int, k: int, p_reuse: float = 0.27) -> np.ndarray:
    """Expert choices [tokens, k] for one layer.  Token 0 draws k distinct
    experts uniformly; for t > 0 slot j keeps token t-1's slot-j expert with
    probability p_reuse, otherwise draws uniformly among experts not yet
    chosen for token t."""
    u = uniform(stream_key(seed, layer, 0, T_TRACE, P_VALUES), tokens * k * 2).reshape(tokens, k, 2)
    out = np.zeros((tokens, k), dtype=np.int32)
    for t in range(tokens):
        chosen: list[int] = []
        keep = [t > 0 and u[t, j, 0] < p_reuse for j in range(k)]
        # kept slots are fixed first so that fresh draws avoid them
        for j in range(k):
            if keep[j]:
                chosen.append(int(out[t - 1, j]))
        for j in range(k):
            if keep[j]:
                out[t, j] = out[t - 1, j]
                continue
            free = np.setdiff1d(np.arange(n_experts), np.asarray(chosen, dtype=np.int64))
            e = int(free[min(int(u[t, j, 1] * len(free)), len(free) - 1)])
            out[t, j] = e
            chosen.append(e)
    return out


def trace_offsets(trace_row: np.ndarray, n_experts: int, boost: float = 30.0) -> np.ndarray:
    """Logit offsets that make the experts of one trace row the top-k."""
    o = np.zeros(n_experts, dtype=np.float32)
    o[np.asarray(trace_row)] = boost
    return o
