"""Operand precision of the tensor-core contraction, checked on the CPU by
emulation against the fp64 oracle (full-width expert, 4 tokens): weights
dequantised once to fp16 (q*s + b rounded once), each activation split into
fp16 hi + lo after a per-token power-of-two scale, fp32 sums.  The expert's
activations and output stay well inside the 2e-3 bar; the same scheme with
bf16 operands does not, which is why the contraction runs kind::f16 with fp16
operands."""
import numpy as np
import pytest

from oracle import moe_oracle as O
from synth import generate as G
from tests.moe_testlib import REL_TOL, rel_err

H, I = 4096, 1024


def _to_f16(x):
    return np.asarray(x, np.float32).astype(np.float16).astype(np.float32)


def _to_bf16(x):
    return G.bf16_bits_to_f32(G.f32_to_bf16_bits(np.asarray(x, np.float32)))


def _contract(W64, X, rnd):
    """D = W X with W rounded once, X [C, T] scaled per token into [2^14, 2^15)
    and split hi + lo, products summed in fp32."""
    Wq = rnd(W64.astype(np.float32))
    X = X.astype(np.float32)
    m = np.max(np.abs(X), axis=0)
    e = np.floor(np.log2(np.where(m > 0, m, 1.0))) - 14
    Xs = X * np.exp2(-e).astype(np.float32)
    hi = rnd(Xs)
    lo = rnd(Xs - hi)
    return ((Wq @ hi).astype(np.float32) + (Wq @ lo).astype(np.float32)) * np.exp2(e).astype(np.float32)


@pytest.fixture(scope="module")
def expert_and_ref():
    ex = G.expert(G.SEED, 0, 3, H, I, 4)
    hs = G.hidden_states(G.SEED, 0, 4, H).astype(np.float64)
    xn = np.stack([O.rmsnorm(h, None, 1e-6) for h in hs], 1)
    wg = O.dequant(*ex["gate"], 4, 64, H)
    wu = O.dequant(*ex["up"], 4, 64, H)
    wd = O.dequant(*ex["down"], 4, 64, I)
    a = O.silu(wg @ xn) * (wu @ xn)
    return (wg, wu, wd, xn), a, wd @ a


def _run(mats, rnd):
    wg, wu, wd, xn = mats
    g = _contract(wg, xn, rnd)
    u = _contract(wu, xn, rnd)
    a = (g / (1.0 + np.exp(-g.astype(np.float64)))) * u
    return a, _contract(wd, a, rnd)


def test_fp16_operands_meet_the_bar(expert_and_ref):
    mats, a_ref, d_ref = expert_and_ref
    a, d = _run(mats, _to_f16)
    for t in range(a.shape[1]):
        assert rel_err(a[:, t], a_ref[:, t]) < 0.25 * REL_TOL
        assert rel_err(d[:, t], d_ref[:, t]) < 0.5 * REL_TOL


def test_bf16_operands_would_not(expert_and_ref):
    mats, a_ref, d_ref = expert_and_ref
    _, d = _run(mats, _to_bf16)
    assert max(rel_err(d[:, t], d_ref[:, t]) for t in range(d.shape[1])) > REL_TOL


def test_fp16_weights_are_nearly_exact():
    """q*s + b from bf16 s, b needs at most 13 significant bits: rounding it to
    fp16 (11 bits) moves most weights by nothing and none by more than 2^-11."""
    codes, s, b = G.matrix(G.SEED, 0, 1, 0, 64, 4096, 4, 64)
    W = O.dequant(codes, s, b, 4, 64, 4096)
    W16 = _to_f16(W).astype(np.float64)
    rel = np.abs(W16 - W) / np.maximum(np.abs(W), 1e-30)
    assert np.max(rel[W != 0]) <= 2.0 ** -11
    assert np.mean(W16 == W) > 0.25
