"""Plain fp64 CPU oracle of the decode-time MoE expert path (test infrastructure).

This file is test infrastructure.  Only the tests, the smoke check and the
benchmark's CPU-baseline leg may import it; the product path never does.  It
shares no code with the CUDA path: it reads the canonical (unpacked) weight
arrays and computes the layer by its plain definition, in float64, one token
at a time, with numpy primitives for unpacking, elementwise maths and the
matrix-vector products.

What it follows (the Flash-MoE pages, quoted by title and section):

* "397B MoE sur MacBook : 4,4 t/s Moteur Flash-MoE", section "Techniques de
  rupture" item 2 and "Flash-MoE - Dizüstünde 397 milyar parametreli modeli
  çalıştırma", section "FMA optimize dequant çekirdeği": a weight is the
  affine dequantisation of an unsigned code, nibble * scale + bias.
* same pages, "Techniques de rupture" item 1 and "Model mimarisi": per layer
  and token, only K = 4 of 512 experts run; one further expert is shared
  (always on).  The routed count K = 4 plus one shared expert, the group size
  64 along the input dimension and bf16 scale/bias are fixed by the workload
  definition, not by the pages.
* "Techniques de rupture" item 4 and "Metal Compute Shaders": the layer is
  RMS norm -> routing -> dequantised matvecs with a fused SwiGLU -> MoE
  combine + residual (+ gate).

Readings where the pages are silent (each listed in the design notes):
* codes are unsigned; element 2j of a row sits in the low nibble of byte j and
  2j+1 in the high nibble (2-bit: element 4j+t in bits 2t..2t+1 of byte j);
* scale/bias group g covers input columns [64g, 64g+64);
* router input and expert input are the RMS-normalised hidden state;
* softmax over all experts, top-K by logit with ties to the lower index,
  weights renormalised over the K chosen (w_k = p_k / sum of chosen p);
* SwiGLU is silu(gate) * up; the shared expert is added with gate 1, or with
  sigmoid(shared_gate . xn) when a shared-gate vector is given;
* y = h + sum_k w_k d_k + g_s d_shared.

Pins: every function here is checked by tests/test_oracle_pins.py against
closed forms, brute force, special cases and the pages' printed sizes.
"""
from __future__ import annotations

import numpy as np


# ----------------------------------------------------------------------------
# storage types
# ----------------------------------------------------------------------------
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> exact float64 values."""
    u32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def unpack_codes(codes: np.ndarray, bits: int, n_cols: int) -> np.ndarray:
    """Unsigned integer codes [rows, n_cols] from packed bytes [rows, n_cols*bits/8].

    Element c of a row is field (c mod 8/bits) of byte c*bits/8, fields counted
    from the least significant bit (reading stated in the module docstring)."""
    codes = np.asarray(codes, dtype=np.uint8)
    per_byte = 8 // bits
    mask = (1 << bits) - 1
    rows = codes.shape[0]
    out = np.empty((rows, codes.shape[1] * per_byte), dtype=np.int64)
    for t in range(per_byte):
        out[:, t::per_byte] = (codes.astype(np.int64) >> (bits * t)) & mask
    return out[:, :n_cols]


def dequant(codes: np.ndarray, scales: np.ndarray, biases: np.ndarray, bits: int,
            group: int, n_cols: int) -> np.ndarray:
    """W[r, c] = q[r, c] * scale[r, c // group] + bias[r, c // group]  (fp64).

    Affine dequantisation "nibble * scale + bias" (page "397B MoE sur MacBook",
    section "Techniques de rupture" item 2)."""
    q = unpack_codes(codes, bits, n_cols).astype(np.float64)
    s = np.repeat(bf16_to_f64(scales), group, axis=1)[:, :n_cols]
    b = np.repeat(bf16_to_f64(biases), group, axis=1)[:, :n_cols]
    return q * s + b


# ----------------------------------------------------------------------------
# layer pieces
# ----------------------------------------------------------------------------
def rmsnorm(h: np.ndarray, gamma_bits: np.ndarray | None, eps: float) -> np.ndarray:
    """xn_i = h_i / sqrt(mean_j h_j^2 + eps) * gamma_i  (gamma = 1 when absent)."""
    h = np.asarray(h, dtype=np.float64)
    r = 1.0 / np.sqrt(np.mean(h * h) + eps)
    g = np.ones_like(h) if gamma_bits is None else bf16_to_f64(gamma_bits)
    return h * r * g


def router_logits(router_bits: np.ndarray, xn: np.ndarray, offset: np.ndarray | None = None) -> np.ndarray:
    """logit_e = sum_i R[e, i] * xn_i (+ offset_e)."""
    logits = bf16_to_f64(router_bits) @ np.asarray(xn, dtype=np.float64)
    if offset is not None:
        logits = logits + np.asarray(offset, dtype=np.float64)
    return logits


def softmax(v: np.ndarray) -> np.ndarray:
    v = np.asarray(v, dtype=np.float64)
    z = np.exp(v - np.max(v))
    return z / np.sum(z)


def topk(logits: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest logits, ordered by (logit desc, index asc)."""
    logits = np.asarray(logits, dtype=np.float64)
    order = np.lexsort((np.arange(logits.size), -logits))
    return order[:k].astype(np.int64)


def routing_weights(logits: np.ndarray, chosen: np.ndarray) -> np.ndarray:
    """Full softmax over all experts, renormalised over the chosen ones."""
    p = softmax(logits)
    pc = p[np.asarray(chosen)]
    return pc / np.sum(pc)


def silu(v: np.ndarray) -> np.ndarray:
    v = np.asarray(v, dtype=np.float64)
    return v / (1.0 + np.exp(-v))


def expert_forward(ex: dict, xn: np.ndarray, hidden: int, inter: int) -> dict:
    """One SwiGLU expert on one token: g = Wg xn, u = Wu xn, a = silu(g) u, d = Wd a."""
    bits, group = ex["bits"], ex["group"]
    wg = dequant(*ex["gate"], bits, group, hidden)
    wu = dequant(*ex["up"], bits, group, hidden)
    wd = dequant(*ex["down"], bits, group, inter)
    xn = np.asarray(xn, dtype=np.float64)
    g = wg @ xn
    u = wu @ xn
    a = silu(g) * u
    d = wd @ a
    return {"g": g, "u": u, "a": a, "d": d}


def layer_decode(h: np.ndarray, *, experts, shared: dict | None, router_bits: np.ndarray,
                 top_k: int, hidden: int, inter: int, eps: float = 1e-6,
                 gamma_bits: np.ndarray | None = None, shared_gate_bits: np.ndarray | None = None,
                 offset: np.ndarray | None = None, force_chosen: np.ndarray | None = None) -> dict:
    """One token through one MoE layer.

    `experts` maps an expert id to its canonical arrays (a dict or a callable,
    so that large layers can be regenerated lazily).  `force_chosen` replaces
    the top-K choice (used to re-run the oracle with another valid choice when
    logits tie)."""
    get = experts if callable(experts) else (lambda e: experts[e])
    h = np.asarray(h, dtype=np.float64)
    xn = rmsnorm(h, gamma_bits, eps)
    logits = router_logits(router_bits, xn, offset)
    chosen = topk(logits, top_k) if force_chosen is None else np.asarray(force_chosen, dtype=np.int64)
    w = routing_weights(logits, chosen)
    d_routed = [expert_forward(get(int(e)), xn, hidden, inter)["d"] for e in chosen]
    y = h.copy()
    for wk, dk in zip(w, d_routed):
        y = y + wk * dk
    out = {"xn": xn, "logits": logits, "chosen": chosen, "w": w, "d_routed": d_routed}
    if shared is not None:
        d_s = expert_forward(shared, xn, hidden, inter)["d"]
        g_s = 1.0
        if shared_gate_bits is not None:
            g_s = 1.0 / (1.0 + np.exp(-(bf16_to_f64(shared_gate_bits) @ xn)))
        y = y + g_s * d_s
        out["d_shared"] = d_s
        out["g_shared"] = g_s
    out["y"] = y
    return out


def tie_margin(logits: np.ndarray, k: int) -> float:
    """Gap between the k-th and (k+1)-th largest logits (inf when k = E)."""
    s = np.sort(np.asarray(logits, dtype=np.float64))[::-1]
    return float("inf") if k >= s.size else float(s[k - 1] - s[k])


def packed_expert_bytes(hidden: int, inter: int, bits: int, group: int = 64) -> int:
    """Bytes of one expert's weights at the given code width: codes for the
    3*H*I weights plus one bf16 scale and one bf16 bias per group."""
    n = 3 * hidden * inter
    return n * bits // 8 + (n // group) * 4
