"""Plant plausible mistakes in the oracle (CPU only, via monkeypatch) and check
that at least one pin fails for each.  This shows the pins can tell a wrong
oracle from a right one."""
import numpy as np
import pytest

import tests.test_oracle_pins as P
from oracle import moe_oracle as O

_orig_dequant = O.dequant
_orig_unpack = O.unpack_codes
_orig_rms = O.rmsnorm
_orig_rw = O.routing_weights
_orig_silu = O.silu
_orig_router = O.router_logits
_orig_expert = O.expert_forward
_orig_layer = O.layer_decode


def _dequant_no_bias(codes, scales, biases, bits, group, n):
    return _orig_dequant(codes, scales, np.zeros_like(biases), bits, group, n)


def _unpack_swapped(codes, bits, n):
    u = _orig_unpack(codes, bits, n)
    per = 8 // bits
    return u.reshape(u.shape[0], -1, per)[:, :, ::-1].reshape(u.shape[0], -1)


def _dequant_shifted_group(codes, scales, biases, bits, group, n):
    return _orig_dequant(codes, np.roll(scales, 1, axis=1), np.roll(biases, 1, axis=1), bits, group, n)


def _rms_eps_outside(h, g, eps):
    h = np.asarray(h, dtype=np.float64)
    r = 1.0 / (np.sqrt(np.mean(h * h)) + eps)
    gg = np.ones_like(h) if g is None else O.bf16_to_f64(g)
    return h * r * gg


def _rw_no_renorm(logits, chosen):
    return O.softmax(logits)[np.asarray(chosen)]


def _silu_neg(v):
    v = np.asarray(v, dtype=np.float64)
    return v / (1.0 + np.exp(v))


def _router_transposed(router_bits, xn, offset=None):
    R = O.bf16_to_f64(router_bits)
    n = min(R.shape)
    lg = R[:n, :n].T @ np.asarray(xn, dtype=np.float64)[:n]
    lg = np.concatenate([lg, np.zeros(R.shape[0] - n)]) if R.shape[0] > n else lg
    return lg if offset is None else lg + offset


def _topk_high_index_ties(logits, k):
    logits = np.asarray(logits, dtype=np.float64)
    order = np.lexsort((-np.arange(logits.size), -logits))
    return order[:k]


def _expert_silu_on_up(ex, xn, hidden, inter):
    out = _orig_expert(ex, xn, hidden, inter)
    a = O.silu(out["u"]) * out["g"]
    wd = O.dequant(*ex["down"], ex["bits"], ex["group"], inter)
    return {**out, "a": a, "d": wd @ a}


def _shared_gate_swapped(out, g_new):
    if "d_shared" not in out:
        return out
    y = out["y"] + (g_new - out["g_shared"]) * out["d_shared"]
    return {**out, "y": y, "g_shared": g_new}


def _layer_gate_sign(h, **kw):
    out = _orig_layer(h, **kw)
    if kw.get("shared_gate_bits") is None:
        return out
    return _shared_gate_swapped(out, 1.0 - out["g_shared"])  # sigmoid(-t) = 1 - sigmoid(t)


def _layer_default_gate_half(h, **kw):
    out = _orig_layer(h, **kw)
    if kw.get("shared_gate_bits") is not None:
        return out
    return _shared_gate_swapped(out, 0.5)


MUTANTS = {
    "dropped bias": ("dequant", _dequant_no_bias),
    "swapped nibble order": ("unpack_codes", _unpack_swapped),
    "shifted group index": ("dequant", _dequant_shifted_group),
    "eps outside sqrt": ("rmsnorm", _rms_eps_outside),
    "no renormalisation": ("routing_weights", _rw_no_renorm),
    "silu sign": ("silu", _silu_neg),
    "router transposed": ("router_logits", _router_transposed),
    "ties to high index": ("topk", _topk_high_index_ties),
    "silu on up": ("expert_forward", _expert_silu_on_up),
    "shared gate sign": ("layer_decode", _layer_gate_sign),
    "default shared gate 0.5": ("layer_decode", _layer_default_gate_half),
}

PINS = [getattr(P, n) for n in dir(P) if n.startswith("test_")]


def _run_pins():
    failures = 0
    for fn in PINS:
        try:
            if "bits" in fn.__code__.co_varnames[: fn.__code__.co_argcount]:
                fn(4)
                fn(2)
            else:
                fn()
        except Exception:  # noqa: BLE001 - any failure counts
            failures += 1
    return failures


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(O, attr, fn)
    assert _run_pins() > 0, f"no pin caught: {name}"


def test_pins_pass_unmutated():
    assert _run_pins() == 0
