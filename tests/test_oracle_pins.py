"""Pins of the fp64 oracle against facts that do not come from the oracle itself:
the pages' printed sizes, closed forms, exact rational brute force, special cases
and invariants.  Each test names the kind of mistake it would catch."""
import itertools
import json
import math
import os
import struct
from fractions import Fraction

import numpy as np
import pytest

from oracle import moe_oracle as O
from synth import generate as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_facts.json")


def facts():
    with open(GOLDEN) as f:
        return json.load(f)


# --------------------------------------------------------------------------- format
def test_expert_size_is_the_pages_6_75_MB():
    """4-bit, group 64, bf16 scale+bias: 3*H*I weights at H=4096, I=1024 give
    exactly the pages' 6.75 MB per expert (a wrong group size or scale dtype
    would not)."""
    f = facts()["expert_size_MB"]
    b = O.packed_expert_bytes(4096, 1024, 4, 64)
    assert b == 7_077_888
    assert b / 2**20 == pytest.approx(f["value"], abs=1e-12)


def test_disk_sizes_consistent_with_pages():
    """60 layers x 512 experts at 4 and 2 bits stay below the pages' 209 GB and
    120 GB totals (GiB reading), which also hold the non-expert weights."""
    f = facts()
    shape = f["model_shape"]
    per4 = O.packed_expert_bytes(shape["hidden"], 1024, 4)
    per2 = O.packed_expert_bytes(shape["hidden"], 1024, 2)
    tot4 = shape["layers"] * shape["experts_per_layer"] * per4 / 2**30
    tot2 = shape["layers"] * shape["experts_per_layer"] * per2 / 2**30
    assert 0.9 * f["disk_GB"]["four_bit"] < tot4 <= f["disk_GB"]["four_bit"]
    assert 0.9 * f["disk_GB"]["two_bit"] < tot2 <= f["disk_GB"]["two_bit"]


# --------------------------------------------------------------------------- storage decoding
def test_bf16_decoding_known_patterns():
    """bf16 bit patterns with textbook values (catches a wrong shift or byte order)."""
    pats = np.array([0x3F80, 0xC000, 0x0000, 0x4049, 0x3C23, 0x8000], dtype=np.uint16)
    want = [1.0, -2.0, 0.0, 3.140625, 0.00994873046875, -0.0]
    got = O.bf16_to_f64(pats)
    assert list(got) == want


def test_unpack_matches_bit_level_reading():
    """Codes read through numpy.unpackbits (an independent route) for both widths."""
    rng = np.random.default_rng(1)
    for bits in (4, 2):
        raw = rng.integers(0, 256, size=(3, 16), dtype=np.uint8)
        n = 16 * 8 // bits
        got = O.unpack_codes(raw, bits, n)
        lsb_bits = np.unpackbits(raw, axis=1, bitorder="little").reshape(3, n, bits)
        want = (lsb_bits * (1 << np.arange(bits))).sum(axis=2)
        assert np.array_equal(got, want)
    # byte 0x21 holds element 0 = 1 (low nibble) and element 1 = 2 (high nibble)
    assert list(O.unpack_codes(np.array([[0x21]], np.uint8), 4, 2)[0]) == [1, 2]
    # byte 0b11100100 holds 2-bit elements 0,1,2,3
    assert list(O.unpack_codes(np.array([[0b11100100]], np.uint8), 2, 4)[0]) == [0, 1, 2, 3]


def _bf16_exact(bits16):
    """Exact rational value of a bf16 pattern via struct (independent of numpy)."""
    (f,) = struct.unpack("<f", struct.pack("<I", int(bits16) << 16))
    return Fraction(f)


@pytest.mark.parametrize("bits", [4, 2])
def test_dequant_matvec_exact_rational_and_fma_rewrite(bits):
    """Brute force in exact rationals on a tiny matrix: the oracle's dequantised
    matvec equals (a) the plain sum of (q*s+b)*x, (b) the pages' FMA rewrite
    fma(q, s*x, b*x) summed, and (c) the group-factored s*sum(q x) + b*sum(x).
    Catches dropped bias, wrong group index and transposition."""
    rng = np.random.default_rng(7 + bits)
    rows, cols, group = 3, 128, 64
    codes = rng.integers(0, 256, size=(rows, cols * bits // 8), dtype=np.uint8)
    sc = S.f32_to_bf16_bits(rng.uniform(0.005, 0.02, size=(rows, cols // group)).astype(np.float32))
    bi = S.f32_to_bf16_bits(rng.uniform(-0.2, 0.0, size=(rows, cols // group)).astype(np.float32))
    # dyadic x so that every product is exact in fp64 too
    x = rng.integers(-64, 64, size=cols) / 16.0
    W = O.dequant(codes, sc, bi, bits, group, cols)
    y = W @ x
    per = 8 // bits
    for r in range(rows):
        q = []
        for byte in codes[r]:
            for t in range(per):
                q.append((int(byte) >> (bits * t)) & ((1 << bits) - 1))
        plain = Fraction(0)
        fma_form = Fraction(0)
        factored = Fraction(0)
        for g in range(cols // group):
            s = _bf16_exact(sc[r, g])
            b = _bf16_exact(bi[r, g])
            sq = Fraction(0)
            sx = Fraction(0)
            for c in range(g * group, (g + 1) * group):
                xc = Fraction(x[c])
                plain += (q[c] * s + b) * xc
                fma_form += q[c] * (s * xc) + (b * xc)
                sq += q[c] * xc
                sx += xc
            factored += s * sq + b * sx
        assert plain == fma_form == factored
        assert abs(Fraction(y[r]) - plain) <= abs(plain) * Fraction(1, 2**50) + Fraction(1, 2**60)


def test_dequant_special_cases():
    """s=1, b=0 gives the integer codes; s=0 gives the bias everywhere; each group
    uses its own (s, b) (a distinct scale per group exposes a shifted group index)."""
    codes = np.array([[0x10, 0x32, 0x54, 0x76] * 16], dtype=np.uint8)  # 128 codes 0..7 repeating
    one = np.full((1, 2), 0x3F80, np.uint16)
    zero = np.zeros((1, 2), np.uint16)
    W = O.dequant(codes, one, zero, 4, 64, 128)
    assert list(W[0, :8]) == [0, 1, 2, 3, 4, 5, 6, 7]
    W = O.dequant(codes, zero, np.array([[0x4000, 0xC040]], np.uint16), 4, 64, 128)
    assert np.all(W[0, :64] == 2.0) and np.all(W[0, 64:] == -3.0)
    W = O.dequant(codes, np.array([[0x3F80, 0x4000]], np.uint16), zero, 4, 64, 128)
    assert W[0, 1] == 1.0 and W[0, 65] == 2.0


# --------------------------------------------------------------------------- rmsnorm
def test_rmsnorm_closed_forms():
    """Hand-computed values, eps placement and gamma (catches eps outside the sqrt,
    sum instead of mean, missing gamma)."""
    assert np.allclose(O.rmsnorm(np.array([3.0, 4.0, 0.0, 0.0]), None, 0.0), [1.2, 1.6, 0.0, 0.0], rtol=0, atol=1e-15)
    assert np.allclose(O.rmsnorm(np.ones(4), None, 3.0), [0.5] * 4, rtol=0, atol=1e-15)
    g = np.array([0x4000, 0x3F80, 0xBF80, 0x0000], np.uint16)  # 2, 1, -1, 0
    assert np.allclose(O.rmsnorm(np.full(4, -7.0), g, 0.0), [-2.0, -1.0, 1.0, 0.0], rtol=0, atol=1e-15)


# --------------------------------------------------------------------------- router / softmax / top-k
def test_router_logits_nonsquare_hand_values():
    """E=2, H=3 router with distinct entries against hand sums (catches a transpose)."""
    R = S.f32_to_bf16_bits(np.array([[1.0, 2.0, 0.5], [-1.0, 0.25, 4.0]], np.float32))
    xn = np.array([1.0, -2.0, 8.0])
    assert list(O.router_logits(R, xn)) == [1.0 - 4.0 + 4.0, -1.0 - 0.5 + 32.0]
    assert list(O.router_logits(R, xn, np.array([10.0, -1.0]))) == [11.0, 29.5]


def test_softmax_known_values():
    p = O.softmax(np.array([0.0, math.log(3.0)]))
    assert p == pytest.approx([0.25, 0.75], abs=1e-15)
    p2 = O.softmax(np.array([1000.0, 1000.0 + math.log(3.0)]))  # shift invariance, no overflow
    assert p2 == pytest.approx([0.25, 0.75], abs=1e-13)  # 1000+ln3 is itself rounded


def _brute_topk(logits, k):
    """The k-subset whose members, listed by (logit desc, index asc), are
    lexicographically largest under (logit, -index)."""
    best, best_key = None, None
    for sub in itertools.combinations(range(len(logits)), k):
        members = sorted(((logits[i], -i) for i in sub), reverse=True)
        if best_key is None or members > best_key:
            best, best_key = [-m[1] for m in members], members
    return best


def test_topk_matches_brute_force_all_subsets():
    """Brute force over all C(E, K) subsets for E <= 12, including hand-built ties."""
    rng = np.random.default_rng(3)
    cases = [rng.normal(size=12) for _ in range(20)]
    cases += [np.round(rng.normal(size=12), 0) for _ in range(20)]  # many exact ties
    cases += [np.zeros(8), np.array([1.0, 2.0, 2.0, 1.0, 2.0, 0.0])]
    for lg in cases:
        for k in (1, 2, 3, 4):
            if k <= lg.size:
                assert list(O.topk(lg, k)) == _brute_topk(list(lg), k)
    assert list(O.topk(np.zeros(16), 4)) == [0, 1, 2, 3]  # zero router -> first K experts


def test_routing_weights_invariants():
    """Weights sum to 1, equal a softmax over the chosen logits only, and do not
    change when one constant is added to every chosen logit (catches a missing
    renormalisation or a softmax over the wrong set)."""
    rng = np.random.default_rng(5)
    lg = rng.normal(size=64) * 1.3
    ch = O.topk(lg, 4)
    w = O.routing_weights(lg, ch)
    assert abs(np.sum(w) - 1.0) < 1e-12
    sel = lg[ch]
    direct = np.exp(sel - sel.max()) / np.exp(sel - sel.max()).sum()
    assert np.allclose(w, direct, rtol=0, atol=1e-15)
    lg2 = lg.copy()
    lg2[ch] += 30.0
    assert list(O.topk(lg2, 4)) == list(ch)
    assert np.allclose(O.routing_weights(lg2, ch), w, rtol=0, atol=1e-13)
    # E == K: weights are the full softmax
    small = rng.normal(size=4)
    assert np.allclose(O.routing_weights(small, O.topk(small, 4)), O.softmax(small)[O.topk(small, 4)], atol=1e-15)


# --------------------------------------------------------------------------- SwiGLU / experts
def test_silu_known_values():
    """silu(0)=0, silu(1)=e/(1+e), odd-part identity silu(x)-silu(-x)=x (catches
    silu(-x) or sigmoid in place of silu)."""
    assert O.silu(np.array([0.0]))[0] == 0.0
    assert O.silu(np.array([1.0]))[0] == pytest.approx(math.e / (1 + math.e), abs=1e-15)
    v = np.linspace(-9, 9, 37)
    assert np.allclose(O.silu(v) - O.silu(-v), v, atol=1e-13)


def _const_matrix(rows, cols, code, s_bits, b_bits, bits=4):
    per = 8 // bits
    byte = 0
    for t in range(per):
        byte |= code << (bits * t)
    codes = np.full((rows, cols * bits // 8), byte, np.uint8)
    return codes, np.full((rows, cols // 64), s_bits, np.uint16), np.full((rows, cols // 64), b_bits, np.uint16)


def test_expert_integer_case_and_zero_gate():
    """s=1, b=0 with integer x: g and u are exact integer matvecs (Python ints).
    A gate that is identically 0 gives a = 0 and d = 0."""
    rng = np.random.default_rng(11)
    H, I = 128, 64
    ex = S.expert(1, 0, 0, H, I, 4)
    one = np.full((I, H // 64), 0x3F80, np.uint16)
    zero = np.zeros((I, H // 64), np.uint16)
    ex["gate"] = (ex["gate"][0], one, zero)
    ex["up"] = (ex["up"][0], one, zero)
    x = rng.integers(-5, 6, size=H).astype(np.float64)
    out = O.expert_forward(ex, x, H, I)
    for r in range(I):
        qg = [(int(b) >> s) & 15 for b in ex["gate"][0][r] for s in (0, 4)]
        qu = [(int(b) >> s) & 15 for b in ex["up"][0][r] for s in (0, 4)]
        assert out["g"][r] == sum(q * int(xi) for q, xi in zip(qg, x))
        assert out["u"][r] == sum(q * int(xi) for q, xi in zip(qu, x))
    ex["gate"] = _const_matrix(I, H, 0, 0x0000, 0x0000)
    out = O.expert_forward(ex, x, H, I)
    assert np.all(out["a"] == 0.0) and np.all(out["d"] == 0.0)


def test_expert_unit_vector_reads_a_column():
    """x = e_j returns column j of the dequantised gate (non-square H != I), so a
    transposed gate would fail."""
    H, I = 192, 64
    ex = S.expert(2, 0, 3, H, I, 4)
    j = 77
    x = np.zeros(H)
    x[j] = 1.0
    out = O.expert_forward(ex, x, H, I)
    codes, sc, bi = ex["gate"]
    col = []
    for r in range(I):
        byte = int(codes[r, j // 2])
        q = (byte >> (4 * (j % 2))) & 15
        col.append(float(_bf16_exact(sc[r, j // 64]) * q + _bf16_exact(bi[r, j // 64])))
    assert np.array_equal(out["g"], np.array(col))


# --------------------------------------------------------------------------- layer
def _tiny_layer(seed=21, H=128, I=64, E=8, bits=4):
    ex = {e: S.expert(seed, 0, e, H, I, bits) for e in range(E)}
    sh = S.expert(seed, 0, S.SHARED_EXPERT, H, I, 4)
    R = S.router(seed, 0, E, H)
    return ex, sh, R


def test_layer_zero_experts_give_residual():
    """All experts output zero (codes 0, s=b=0): y == h exactly (catches a missing
    or doubled residual)."""
    H, I, E = 128, 64, 8
    ex, sh, R = _tiny_layer(H=H, I=I, E=E)
    z = {"bits": 4, "group": 64, "gate": _const_matrix(I, H, 0, 0, 0), "up": _const_matrix(I, H, 0, 0, 0),
         "down": _const_matrix(H, I, 0, 0, 0)}
    h = S.hidden_states(1, 0, 1, H)[0].astype(np.float64)
    out = O.layer_decode(h, experts={e: z for e in range(E)}, shared=z, router_bits=R, top_k=4, hidden=H, inter=I)
    assert np.array_equal(out["y"], h)


def test_layer_linear_in_weights_and_shared_gate():
    """y - h equals sum_k w_k d_k + g_s d_s computed from separately evaluated
    experts; a zero shared-gate vector gives g_s = 1/2 (sigmoid(0))."""
    H, I, E = 128, 64, 8
    ex, sh, R = _tiny_layer(H=H, I=I, E=E)
    h = S.hidden_states(2, 0, 1, H)[0].astype(np.float64)
    out = O.layer_decode(h, experts=ex, shared=sh, router_bits=R, top_k=4, hidden=H, inter=I,
                         shared_gate_bits=np.zeros(H, np.uint16))
    assert out["g_shared"] == 0.5
    xn = out["xn"]
    acc = h.copy()
    for k, e in enumerate(out["chosen"]):
        acc += out["w"][k] * O.expert_forward(ex[int(e)], xn, H, I)["d"]
    acc += 0.5 * O.expert_forward(sh, xn, H, I)["d"]
    assert np.allclose(out["y"], acc, rtol=0, atol=1e-12)
    assert abs(out["w"].sum() - 1.0) < 1e-12


def test_packed_bytes_tiny_and_two_bit():
    assert O.packed_expert_bytes(256, 128, 4) == 55_296
    assert O.packed_expert_bytes(4096, 1024, 2) == 3_932_160
    assert O.packed_expert_bytes(256, 128, 2) == 30_720


# --------------------------------------------------------------------------- SwiGLU order and the shared gate
def _unit_expert(H, I, gate_code, up_code):
    """An expert whose gate and up rows all dequantise to the integer codes
    given (scale 1, bias 0), so that g and u are known sums of x."""
    one = np.full((I, H // 64), 0x3F80, np.uint16)
    zero = np.zeros((I, H // 64), np.uint16)
    ex = {"bits": 4, "group": 64}
    ex["gate"] = (_const_matrix(I, H, gate_code, 0x3F80, 0)[0], one, zero)
    ex["up"] = (_const_matrix(I, H, up_code, 0x3F80, 0)[0], one, zero)
    ex["down"] = _const_matrix(H, I, 1, 0x3F80, 0)
    return ex


def test_swiglu_is_silu_of_gate_times_up():
    """SwiGLU order ("397B MoE sur MacBook", "Techniques de rupture" item 4: the
    fused SwiGLU): a = silu(g) * u, not silu(u) * g.  With x = e_0 the gate rows
    give g = 1 and the up rows u = 2, so every a must be 2 * sigmoid(1) =
    2e / (1 + e) = 1.4621..., while the swapped order would give
    silu(2) = 2 / (1 + e^-2) = 1.7616...  Also: a is linear in u (doubling the
    up codes doubles a exactly) but not in g."""
    H, I = 64, 64
    x = np.zeros(H)
    x[0] = 1.0
    out = O.expert_forward(_unit_expert(H, I, 1, 2), x, H, I)
    assert np.all(out["g"] == 1.0) and np.all(out["u"] == 2.0)
    assert np.allclose(out["a"], 2.0 * math.e / (1.0 + math.e), rtol=0, atol=1e-15)
    assert not np.allclose(out["a"], 2.0 / (1.0 + math.exp(-2.0)), rtol=0, atol=1e-3)
    # the down rows (all codes 1, scale 1) sum the 64 activations
    assert np.allclose(out["d"], 64 * 2.0 * math.e / (1.0 + math.e), rtol=0, atol=1e-12)
    a_u4 = O.expert_forward(_unit_expert(H, I, 1, 4), x, H, I)["a"]
    a_g2 = O.expert_forward(_unit_expert(H, I, 2, 2), x, H, I)["a"]
    assert np.allclose(a_u4, 2.0 * out["a"], rtol=0, atol=1e-15)
    assert not np.allclose(a_g2, 2.0 * out["a"], rtol=0, atol=1e-3)


def _gate_layer_case(shared_gate_bits):
    """A tiny layer with h = 1 everywhere and eps = 0, so xn = 1 exactly, and a
    shared expert whose output is known: gate codes 1, up codes 1 give g = u = H
    per row, a = silu(H) * H; the down rows sum the activations."""
    H, I, E = 128, 64, 8
    ex, _, R = _tiny_layer(H=H, I=I, E=E)
    sh = _unit_expert(H, I, 1, 1)
    h = np.ones(H)
    out = O.layer_decode(h, experts=ex, shared=sh, router_bits=R, top_k=4, hidden=H, inter=I, eps=0.0,
                         shared_gate_bits=shared_gate_bits)
    a = H / (1.0 + math.exp(-H)) * H
    d_s = np.full(H, I * a)
    routed = sum(out["w"][k] * O.expert_forward(ex[int(e)], np.ones(H), H, I)["d"] for k, e in enumerate(out["chosen"]))
    return out, h, d_s, routed


def test_shared_gate_is_sigmoid_of_gate_dot_xn():
    """The "gate" of "MoE combine + residual + gate" ("Flash-MoE - Dizüstünde
    ...", "Metal Compute Shaders"), read as g_s = sigmoid(shared_gate . xn).
    With xn = 1 and a gate vector whose only nonzero entries are +2 and -0.5,
    shared_gate . xn = 1.5 and g_s = 1 / (1 + e^-1.5) = 0.8175744762; the
    opposite sign would give 0.1824255238.  y - h - (routed part) must be
    g_s times the shared expert's output."""
    g = np.zeros(128, np.uint16)
    g[5] = 0x4000   # +2.0
    g[77] = 0xBF00  # -0.5
    out, h, d_s, routed = _gate_layer_case(g)
    assert out["g_shared"] == pytest.approx(0.8175744761936437, abs=1e-15)
    assert np.allclose(out["y"] - h - routed, 0.8175744761936437 * d_s, rtol=1e-13, atol=0)


def test_shared_expert_default_gate_is_one():
    """Without a shared-gate vector the shared expert is added as it is
    (g_s = 1): y - h - (routed part) equals its output exactly."""
    out, h, d_s, routed = _gate_layer_case(None)
    assert out["g_shared"] == 1.0
    assert np.allclose(out["y"] - h - routed, d_s, rtol=1e-13, atol=0)
