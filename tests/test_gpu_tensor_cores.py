"""Parity of the batched tensor-core contraction (MOE_TENSOR_CORES) with the
fp64 oracle, through moe_expert_forward and moe_layer_decode: one expert on
three tokens (tiny, odd and full-width shapes, 4- and 2-bit), the tiny layer
at B = 2, chunks of more than kTcTok = 32 entries, a ragged last code stage
and row tile, no shared expert, gamma and shared gate, 2-bit routed experts,
the full-width layer with skewed routing (every token of B = 8 and 64, and
equality of the routing with the dp4a path)."""
import numpy as np
import pytest

from synth import generate as G
from tests.moe_testlib import REL_TOL, build_layer, rel_err, routing_ok, workspace

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import bit_expert_matvec_moe_b300 as M  # noqa: E402

TINY = dict(hidden=256, inter=128, n_experts=16, top_k=4)
FULL = dict(hidden=4096, inter=1024, n_experts=512, top_k=4)


def D(shape, bits=4, flags=M.MOE_HAS_SHARED, **kw):
    d = dict(shape)
    d.update(kw)
    return M.Dims(bits=bits, flags=flags, **d)


@pytest.fixture(scope="module", autouse=True)
def _build():
    from bit_expert_matvec_moe_b300 import build
    from synth import device

    build.build()
    device.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def decode_tc(L, h_np, offset=None, tc=True):
    B = h_np.shape[0]
    d = L.dims
    d = M.Dims(**{**d.__dict__, "flags": d.flags | (M.MOE_TENSOR_CORES if tc else 0)})
    layer = M.make_layer(d, L.experts, L.stride, L.router, shared=L.shared, shared_bits=L.shared_bits,
                         rms_gamma=L.gamma, shared_gate=L.gate)
    h = torch.from_numpy(np.ascontiguousarray(h_np, dtype=np.float32)).cuda()
    idx = torch.empty((B, d.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((B, d.top_k), dtype=torch.float32, device="cuda")
    off = None if offset is None else torch.from_numpy(np.ascontiguousarray(offset, dtype=np.float32)).cuda()
    ws = workspace(d, B)
    M.moe_layer_decode(layer, h, ws, logit_offset=off, idx_out=idx, w_out=w)
    st = M.moe_get_device_status(ws)
    assert st == 0, f"device status {st}"
    return h.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()


def check(L, h_tok, y, idx, w, offset=None, ref=None, delta_tol=REL_TOL):
    ref = L.oracle(h_tok, offset=offset) if ref is None else ref
    ok, tie = routing_ok(idx, ref["logits"], L.dims.top_k)
    assert ok
    if tie:
        ref = L.oracle(h_tok, offset=offset, force_chosen=idx)
    assert rel_err(y, ref["y"]) <= REL_TOL, rel_err(y, ref["y"])
    assert rel_err(y - h_tok, ref["y"] - h_tok) <= delta_tol, rel_err(y - h_tok, ref["y"] - h_tok)


@pytest.mark.parametrize("bits", [4, 2])
@pytest.mark.parametrize("shape", [TINY, FULL, dict(hidden=320, inter=64, n_experts=4, top_k=2)])
def test_tc_expert_forward(bits, shape):
    """One expert on B = 3 tokens through moe_expert_forward: each token's
    expert output against the oracle, overwrite and weighted accumulate."""
    from oracle import moe_oracle as O
    from tests.moe_testlib import pack_expert_device

    d = D(shape, bits=bits, flags=M.MOE_TENSOR_CORES)
    H, I, B = d.hidden, d.inter, 3
    canon = G.expert(G.SEED, 2, 9, H, I, bits)
    blob = torch.empty(M.moe_packed_expert_bytes(d, bits), dtype=torch.uint8, device="cuda")
    pack_expert_device(d, bits, canon, blob, torch)
    xn = G.hidden_states(G.SEED, 2, B, H)
    base = G.hidden_states(G.SEED, 3, B, H)
    row_w = np.array([0.5, -1.25, 2.0], np.float32)
    ws = workspace(d, B)
    out = torch.from_numpy(base.copy()).cuda()
    M.moe_expert_forward(d, bits, blob, torch.from_numpy(xn).cuda(), out, ws,
                         row_w=torch.from_numpy(row_w).cuda(), accumulate=True)
    out2 = torch.zeros((B, H), dtype=torch.float32, device="cuda")
    M.moe_expert_forward(d, bits, blob, torch.from_numpy(xn).cuda(), out2, ws)
    assert M.moe_get_device_status(ws) == 0
    out, out2 = out.cpu().numpy(), out2.cpu().numpy()
    for b in range(B):
        ref = O.expert_forward(canon, xn[b], H, I)["d"]
        assert rel_err(out2[b], ref) <= REL_TOL, rel_err(out2[b], ref)
        assert rel_err(out[b], base[b] + row_w[b] * ref) <= REL_TOL


def test_tc_tiny_two_tokens():
    L = build_layer(D(TINY))
    h = G.hidden_states(G.SEED, 40, 2, 256)
    y, idx, w = decode_tc(L, h)
    for t in range(2):
        check(L, h[t], y[t], idx[t], w[t])


@pytest.mark.parametrize("bits", [4, 2])
def test_tc_tiny_many_tokens_per_expert(bits):
    """33 tokens all routed to the same 4 experts: every expert (and the shared
    one) has a chunk of 32 entries and a chunk of 1."""
    L = build_layer(D(TINY, bits=bits), shared_bits=bits)
    B = 33
    h = G.hidden_states(G.SEED, 41, B, 256)
    off = np.zeros((B, 16), np.float32)
    off[:, [2, 5, 11, 13]] = 30.0
    y, idx, w = decode_tc(L, h, offset=off)
    assert all(sorted(r) == [2, 5, 11, 13] for r in idx.tolist())
    for t in (0, 31, 32):
        check(L, h[t], y[t], idx[t], w[t], offset=off[t])


@pytest.mark.parametrize("variant", ["odd_shape", "no_shared", "gamma_gate"])
def test_tc_edge_shapes(variant):
    if variant == "odd_shape":  # 5 groups along hidden (ragged code stage), 320 down rows (ragged row tile)
        L = build_layer(D(dict(hidden=320, inter=64, n_experts=4, top_k=2)))
        H = 320
    elif variant == "no_shared":
        L = build_layer(D(TINY, flags=0))
        H = 256
    else:
        L = build_layer(D(TINY, flags=M.MOE_HAS_SHARED | M.MOE_HAS_SHARED_GATE), gamma=True, shared_gate=True)
        H = 256
    h = G.hidden_states(G.SEED, 42, 6, H)
    y, idx, w = decode_tc(L, h)
    for t in (0, 5):
        check(L, h[t], y[t], idx[t], w[t])


@pytest.mark.parametrize("bits", [4, 2])
def test_tc_odd_group_counts_many_units(bits):
    """5 groups along hidden and 3 along inter, 64 experts and 64 tokens: more
    units than CTAs, so a CTA's K-block count crosses odd unit boundaries (the
    dequantising warps split K-blocks by their parity over the whole launch)."""
    d = D(dict(hidden=320, inter=192, n_experts=64, top_k=4), bits=bits)
    L = build_layer(d, shared_bits=bits)
    B = 64
    h = G.hidden_states(G.SEED, 45, B, 320)
    y, idx, w = decode_tc(L, h)
    y2, idx2, w2 = decode_tc(L, h, tc=False)
    assert (idx == idx2).all()
    refs = L.oracle_many(h)
    # The layer output meets the bar; its MoE part alone (output minus the
    # residual) gets 4e-3 at 2 bits: the A operand holds each weight q*s + b
    # rounded to fp16 (relative 2^-11) and a 320-input sum averages few of them.
    delta_tol = REL_TOL if bits == 4 else 4e-3
    for t in range(B):
        check(L, h[t], y[t], idx[t], w[t], ref=refs[t], delta_tol=delta_tol)


@pytest.mark.parametrize("B", [8, 64])
def test_tc_full_width_skewed(B):
    L = build_layer(D(FULL), gen="device")
    h = G.hidden_states(G.SEED, 43, B, 4096)
    off = np.tile(G.popularity_offsets(G.SEED, 0, 512), (B, 1))
    y, idx, w = decode_tc(L, h, offset=off)
    y2, idx2, w2 = decode_tc(L, h, offset=off, tc=False)
    assert (idx == idx2).all()  # routing does not depend on the contraction
    assert rel_err(y, y2) <= REL_TOL
    refs = L.oracle_many(h, offset=off)
    for t in range(B):
        check(L, h[t], y[t], idx[t], w[t], offset=off[t], ref=refs[t])


def test_tc_two_bit_full_width():
    L = build_layer(D(FULL, bits=2), gen="device")
    h = G.hidden_states(G.SEED, 44, 8, 4096)
    y, idx, w = decode_tc(L, h)
    refs = L.oracle_many(h)
    for t in range(8):
        check(L, h[t], y[t], idx[t], w[t], ref=refs[t])
