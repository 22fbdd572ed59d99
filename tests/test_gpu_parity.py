"""Parity of the CUDA path (through the C ABI) with the fp64 oracle on the same
seeded inputs.  Bar: routing indices exact (up to oracle-logit ties within
1e-6), floating outputs within max relative error 2e-3 (floor 1e-3 of the
largest magnitude), integer/byte work bit-exact."""
import numpy as np
import pytest

from oracle import moe_oracle as O
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


@pytest.fixture(scope="module")
def full4():
    return build_layer(D(FULL), gen="device")


def decode(L, h_np, offset=None, flags_extra=0, ws=None):
    """Run moe_layer_decode on tokens h_np [B, H]; returns (y, idx, w)."""
    B = h_np.shape[0]
    d = L.dims
    if flags_extra:
        d = M.Dims(**{**d.__dict__, "flags": d.flags | flags_extra})
    layer = M.make_layer(d, L.experts, L.stride, L.router, shared=L.shared, shared_bits=L.shared_bits,
                         rms_gamma=L.gamma, shared_gate=L.gate)
    h = torch.from_numpy(np.ascontiguousarray(h_np, dtype=np.float32)).cuda()
    idx = torch.empty((B, d.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((B, d.top_k), dtype=torch.float32, device="cuda")
    off = None if offset is None else torch.from_numpy(np.ascontiguousarray(offset, dtype=np.float32)).cuda()
    ws = ws if ws is not None else workspace(d, B)
    M.moe_layer_decode(layer, h, ws, logit_offset=off, idx_out=idx, w_out=w)
    st = M.moe_get_device_status(ws)
    assert st == 0, f"device status {st}"
    return h.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()


def check_token(L, h_tok, y, idx, w, offset=None, ref=None):
    ref = L.oracle(h_tok, offset=offset) if ref is None else ref
    ok, tie = routing_ok(idx, ref["logits"], L.dims.top_k)
    assert ok, (idx, O.topk(ref["logits"], L.dims.top_k))
    if tie:
        ref = L.oracle(h_tok, offset=offset, force_chosen=idx)
    assert rel_err(w, ref["w"]) <= REL_TOL
    assert abs(float(np.sum(w)) - 1.0) < 1e-5
    assert rel_err(y, ref["y"]) <= REL_TOL, rel_err(y, ref["y"])
    assert rel_err(y - h_tok, ref["y"] - h_tok) <= REL_TOL, rel_err(y - h_tok, ref["y"] - h_tok)
    return ref


def check_batch(L, h, y, idx, w, offset=None):
    """Every token of a batch against the oracle (each touched expert
    dequantised once for all of its tokens)."""
    refs = L.oracle_many(h, offset=offset)
    for t in range(h.shape[0]):
        check_token(L, h[t], y[t], idx[t], w[t], offset=None if offset is None else offset[t], ref=refs[t])


# --------------------------------------------------------------------------- generator + packing
def test_device_generator_matches_host():
    from synth import device as SD

    for (rows, cols, bits, t) in [(128, 256, 4, G.T_GATE), (4096, 1024, 2, G.T_DOWN), (64, 192, 4, G.T_UP)]:
        c, s, b = SD.matrix(G.SEED, 3, 7, t, rows, cols, bits)
        hc, hs, hb = G.matrix(G.SEED, 3, 7, t, rows, cols, bits, 64)
        assert np.array_equal(c.cpu().numpy(), hc)
        assert np.array_equal(s.cpu().numpy().view(np.uint16), hs)
        assert np.array_equal(b.cpu().numpy().view(np.uint16), hb)


def unpack_row_codes(packed, bits, ng):
    """Canonical code bytes of one row from the packed order (host parser
    written from the layout description, independent of the pack kernel).
    4-bit: groups in chunks of up to 32; in a chunk of n groups, the first
    16-byte halves of all n groups, then all second halves.
    2-bit: field t of byte j of word m holds input 16m + (2j, 2j+1, 8+2j, 9+2j)[t]."""
    packed = np.asarray(packed, dtype=np.uint8)
    if bits == 4:
        out = np.empty(32 * ng, np.uint8)
        for g in range(ng):
            k, i = divmod(g, 32)
            n = min(32, ng - 32 * k)
            for h in range(2):
                src = 1024 * k + 16 * (h * n + i)
                out[32 * g + 16 * h:32 * g + 16 * h + 16] = packed[src:src + 16]
        return out
    nwords = packed.size // 4
    vals = np.zeros(16 * nwords, np.int64)  # input index -> 2-bit code
    for m in range(nwords):
        w = int.from_bytes(packed[4 * m:4 * m + 4].tobytes(), "little")
        for j in range(4):
            for t, u in enumerate((2 * j, 2 * j + 1, 8 + 2 * j, 9 + 2 * j)):
                vals[16 * m + u] = (w >> (8 * j + 2 * t)) & 3
    canon = np.zeros(4 * nwords, np.uint8)
    for c in range(16 * nwords):
        canon[c // 4] |= np.uint8(vals[c] << (2 * (c % 4)))
    return canon


@pytest.mark.parametrize("bits", [4, 2])
@pytest.mark.parametrize("shape", [TINY, dict(hidden=320, inter=64, n_experts=4, top_k=2),
                                   dict(hidden=3072, inter=128, n_experts=4, top_k=2)])
def test_pack_layout_bit_exact(bits, shape):
    """Read the packed blob back with an independent host parser."""
    from tests.moe_testlib import pack_expert_device

    d = D(shape, bits=bits)
    H, I = d.hidden, d.inter
    canon = G.expert(G.SEED, 0, 1, H, I, bits)
    n = M.moe_packed_expert_bytes(d, bits)
    dst = torch.full((n,), 0xAB, dtype=torch.uint8, device="cuda")
    pack_expert_device(d, bits, canon, dst, torch)
    blob = dst.cpu().numpy()

    def pad16(x):
        return (x + 15) // 16 * 16

    gu_codes, d_codes = H * bits // 8, I * bits // 8
    gu_row, d_row = pad16(gu_codes + 4 * (H // 64)), pad16(d_codes + 4 * (I // 64))
    assert n == I * 2 * gu_row + H * d_row
    rows_to_check = sorted({0, 1, I // 2, I - 1})
    for r in rows_to_check:
        for m, name in enumerate(("gate", "up")):
            row = blob[r * 2 * gu_row + m * gu_row:][:gu_row]
            c, s, b = canon[name]
            assert np.array_equal(unpack_row_codes(row[:gu_codes], bits, H // 64), c[r])
            sb = row[gu_codes:gu_codes + 4 * (H // 64)].view(np.uint16).reshape(-1, 2)
            assert np.array_equal(sb[:, 0], s[r]) and np.array_equal(sb[:, 1], b[r])
            assert np.all(row[gu_codes + 4 * (H // 64):] == 0)
    base = I * 2 * gu_row
    c, s, b = canon["down"]
    for j in sorted({0, 1, H // 2, H - 1}):
        row = blob[base + j * d_row:][:d_row]
        assert np.array_equal(unpack_row_codes(row[:d_codes], bits, I // 64), c[j])
        sb = row[d_codes:d_codes + 4 * (I // 64)].view(np.uint16).reshape(-1, 2)
        assert np.array_equal(sb[:, 0], s[j]) and np.array_equal(sb[:, 1], b[j])
        assert np.all(row[d_codes + 4 * (I // 64):] == 0)


# --------------------------------------------------------------------------- routing
@pytest.mark.parametrize("shape", [TINY, FULL])
@pytest.mark.parametrize("B", [1, 5])
@pytest.mark.parametrize("with_offset", [False, True])
def test_route_parity(shape, B, with_offset):
    d = D(shape)
    E, H, K = d.n_experts, d.hidden, d.top_k
    R = G.router(G.SEED, 11, E, H)
    xn = G.hidden_states(G.SEED, 11, B, H)
    off = np.stack([G.popularity_offsets(G.SEED, 11 + b, E) for b in range(B)]) if with_offset else None
    ws = workspace(d, B)
    idx = torch.empty((B, K), dtype=torch.int32, device="cuda")
    w = torch.empty((B, K), dtype=torch.float32, device="cuda")
    lg = torch.empty((B, E), dtype=torch.float32, device="cuda")
    M.moe_route(d, torch.from_numpy(xn).cuda(), torch.from_numpy(R.view(np.int16)).cuda(), idx, w, ws,
                logit_offset=None if off is None else torch.from_numpy(off).cuda(), logits_out=lg)
    assert M.moe_get_device_status(ws) == 0
    idx, w, lg = idx.cpu().numpy(), w.cpu().numpy(), lg.cpu().numpy()
    for b in range(B):
        ref_lg = O.router_logits(R, xn[b], None if off is None else off[b])
        assert rel_err(lg[b], ref_lg) <= REL_TOL
        assert np.max(np.abs(lg[b] - ref_lg)) < 1e-5
        ok, tie = routing_ok(idx[b], ref_lg, K)
        assert ok
        chosen = idx[b] if tie else O.topk(ref_lg, K)
        assert rel_err(w[b], O.routing_weights(ref_lg, chosen)) <= REL_TOL


def test_route_exact_ties_take_lower_index():
    d = D(TINY)
    R = np.zeros((16, 256), np.uint16)
    xn = G.hidden_states(G.SEED, 0, 2, 256)
    ws = workspace(d, 2)
    idx = torch.empty((2, 4), dtype=torch.int32, device="cuda")
    w = torch.empty((2, 4), dtype=torch.float32, device="cuda")
    M.moe_route(d, torch.from_numpy(xn).cuda(), torch.from_numpy(R.view(np.int16)).cuda(), idx, w, ws)
    assert idx.cpu().numpy().tolist() == [[0, 1, 2, 3], [0, 1, 2, 3]]
    assert np.allclose(w.cpu().numpy(), 0.25, atol=1e-7)


# --------------------------------------------------------------------------- one expert
@pytest.mark.parametrize("bits", [4, 2])
@pytest.mark.parametrize("shape", [TINY, FULL, dict(hidden=320, inter=64, n_experts=4, top_k=2)])
def test_expert_forward_parity(bits, shape):
    from tests.moe_testlib import pack_expert_device

    d = D(shape, bits=bits)
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


# --------------------------------------------------------------------------- whole layer
PATH_FLAGS = {"fused": 0, "fused_pdl": M.MOE_PDL, "multi": M.MOE_NO_FUSED}


@pytest.mark.parametrize("path", ["fused", "fused_pdl", "multi"])
def test_layer_tiny(path):
    L = build_layer(D(TINY))
    h = G.hidden_states(G.SEED, 0, 6, 256)
    for t in range(6):
        y, idx, w = decode(L, h[t:t + 1], flags_extra=PATH_FLAGS[path])
        check_token(L, h[t], y[0], idx[0], w[0])


@pytest.mark.parametrize("path", ["fused", "fused_pdl", "multi"])
def test_layer_full_width(full4, path):
    h = G.hidden_states(G.SEED, 0, 3, 4096)
    for t in range(3 if path != "multi" else 1):
        y, idx, w = decode(full4, h[t:t + 1], flags_extra=PATH_FLAGS[path])
        check_token(full4, h[t], y[0], idx[0], w[0])


def test_pdl_back_to_back_calls_match_oracle(full4):
    """Many single-token calls queued back to back with programmatic dependent
    launch, each call reading the h the previous call wrote (a chain), so that a
    kernel that read h before the previous one finished would diverge."""
    d = M.Dims(**{**full4.dims.__dict__, "flags": full4.dims.flags | M.MOE_PDL})
    layer = M.make_layer(d, full4.experts, full4.stride, full4.router, shared=full4.shared, shared_bits=4)
    h0 = G.hidden_states(G.SEED, 21, 1, 4096)
    h = torch.from_numpy(h0.copy()).cuda()
    ws = workspace(d, 1)
    n = 6
    for _ in range(n):
        M.moe_layer_decode(layer, h, ws)
    assert M.moe_get_device_status(ws) == 0
    ref = h0[0].astype(np.float64)
    for _ in range(n):
        ref = full4.oracle(ref)["y"]
    assert rel_err(h.cpu().numpy()[0], ref) <= REL_TOL


@pytest.mark.parametrize("tc", [False, True])
def test_pdl_batched_chain_matches_plain_launches(full4, tc):
    """Batched calls (B = 8) queued back to back with every kernel of the
    multi-kernel path chained by programmatic dependent launch, each call
    reading the h the previous call wrote: the results equal those of plain
    launches bit for bit (same kernels, same order of arithmetic), and the
    first call matches the oracle at every token."""
    B, n = 8, 3
    h0 = G.hidden_states(G.SEED, 22, B, 4096)
    off = np.tile(G.popularity_offsets(G.SEED, 0, 512), (B, 1))
    extra = M.MOE_TENSOR_CORES if tc else 0
    outs = {}
    for pdl in (False, True):
        d = M.Dims(**{**full4.dims.__dict__, "flags": full4.dims.flags | extra | (M.MOE_PDL if pdl else 0)})
        layer = M.make_layer(d, full4.experts, full4.stride, full4.router, shared=full4.shared, shared_bits=4)
        h = torch.from_numpy(h0.copy()).cuda()
        o = torch.from_numpy(off).cuda()
        ws = workspace(d, B)
        idx = torch.empty((B, 4), dtype=torch.int32, device="cuda")
        w = torch.empty((B, 4), dtype=torch.float32, device="cuda")
        ys = []
        for c in range(n):
            M.moe_layer_decode(layer, h, ws, logit_offset=o, idx_out=idx if c == 0 else None,
                               w_out=w if c == 0 else None)
            ys.append(h.clone())
        assert M.moe_get_device_status(ws) == 0
        outs[pdl] = ([y.cpu().numpy() for y in ys], idx.cpu().numpy(), w.cpu().numpy())
    for a, b in zip(outs[False][0], outs[True][0]):
        assert np.array_equal(a, b)
    assert np.array_equal(outs[False][1], outs[True][1])
    check_batch(full4, h0, outs[True][0][0], outs[True][1], outs[True][2], offset=off)


def test_fused_is_deterministic(full4):
    h = G.hidden_states(G.SEED, 5, 1, 4096)
    y1, i1, w1 = decode(full4, h)
    y2, i2, w2 = decode(full4, h)
    assert np.array_equal(y1, y2) and np.array_equal(i1, i2) and np.array_equal(w1, w2)


@pytest.mark.parametrize("B", [8, 32, 128])
def test_layer_batched_full_width_skewed(full4, B):
    """Batched decode with per-expert popularity offsets (the batched sweep's
    routing): tokens share experts, and every token must equal its own oracle
    result.  B = 32 and 128 split the shared expert into several work items."""
    h = G.hidden_states(G.SEED, 7, B, 4096)
    off = np.tile(G.popularity_offsets(G.SEED, 0, 512), (B, 1))
    y, idx, w = decode(full4, h, offset=off)
    assert len(np.unique(idx)) < B * 4  # experts are shared inside the batch
    check_batch(full4, h, y, idx, w, offset=off)


@pytest.mark.parametrize("B", [1, 8])
def test_layer_two_bit_full_width(B):
    """2-bit routed experts with the 4-bit shared expert."""
    L = build_layer(D(FULL, bits=2), gen="device")
    h = G.hidden_states(G.SEED, 9, B, 4096)
    y, idx, w = decode(L, h)
    check_batch(L, h, y, idx, w)


@pytest.mark.parametrize("path", ["fused", "fused_pdl", "multi"])
@pytest.mark.parametrize("variant", ["gamma_gate", "no_shared", "e_equals_k", "k1", "odd_shape", "stride_pad",
                                     "two_bit_tiny"])
def test_layer_edge_cases(path, variant):
    shape, kw, bkw = dict(TINY), {}, {}
    if variant == "gamma_gate":
        kw["flags"] = M.MOE_HAS_SHARED | M.MOE_HAS_SHARED_GATE
        bkw = dict(gamma=True, shared_gate=True)
    elif variant == "no_shared":
        kw["flags"] = 0
    elif variant == "e_equals_k":
        shape.update(n_experts=4, top_k=4)
    elif variant == "k1":
        shape.update(top_k=1)
    elif variant == "odd_shape":
        shape = dict(hidden=320, inter=64, n_experts=24, top_k=3)
    elif variant == "stride_pad":
        bkw = dict(stride_pad=256)
    elif variant == "two_bit_tiny":
        kw["bits"] = 2
        bkw = dict(shared_bits=2)
    L = build_layer(D(shape, **kw), **bkw)
    h = G.hidden_states(G.SEED, 4, 3, L.dims.hidden)
    for t in range(3):
        y, idx, w = decode(L, h[t:t + 1], flags_extra=PATH_FLAGS[path])
        check_token(L, h[t], y[0], idx[0], w[0])


def test_workspace_reused_across_shapes():
    """One workspace serves layers of different top-K and with and without a
    shared expert, in turn: the grid barriers of the single-token kernel must
    stay in step whichever subset a call uses."""
    L4 = build_layer(D(TINY))
    L2 = build_layer(D(TINY, top_k=2))
    L0 = build_layer(D(TINY, flags=0))
    big = M.Dims(**{**L4.dims.__dict__, "top_k": 8})
    ws = workspace(big, 1)
    h = G.hidden_states(G.SEED, 31, 6, 256)
    for t, L in enumerate([L4, L2, L4, L0, L2, L4]):
        y, idx, w = decode(L, h[t:t + 1], ws=ws)
        check_token(L, h[t], y[0], idx[0], w[0])


def test_layer_batch_edges():
    """B = 1..B_max through the multi-kernel path, and a batch whose tokens all
    pick the same experts (one work item per expert)."""
    L = build_layer(D(TINY))
    h = G.hidden_states(G.SEED, 12, 33, 256)
    y, idx, w = decode(L, h)
    check_batch(L, h, y, idx, w)
    off = np.zeros((16, 16), np.float32)
    off[:, [3, 7, 9, 12]] = 30.0
    hs = G.hidden_states(G.SEED, 13, 16, 256)
    y, idx, w = decode(L, hs, offset=off)
    assert all(sorted(r) == [3, 7, 9, 12] for r in idx.tolist())
    check_batch(L, hs, y, idx, w, offset=off)


# --------------------------------------------------------------------------- device status
def test_nonfinite_input_sets_status():
    L = build_layer(D(TINY))
    for flags_extra in (0, M.MOE_NO_FUSED):
        d = M.Dims(**{**L.dims.__dict__, "flags": L.dims.flags | flags_extra})
        layer = M.make_layer(d, L.experts, L.stride, L.router, shared=L.shared)
        h = torch.from_numpy(G.hidden_states(G.SEED, 1, 1, 256)).cuda()
        h[0, 3] = float("nan")
        ws = workspace(d, 1)
        M.moe_layer_decode(layer, h, ws)
        assert M.moe_get_device_status(ws) == 5  # MOE_ERR_NONFINITE
        assert M.moe_get_device_status(ws) == 0  # cleared by the read


def test_barrier_timeout_is_reported_and_recoverable():
    """Cross-block waits that expect a later launch's data never complete (the
    workspace test hook): every block gives up after its bounded wait, the
    status word says TIMEOUT, later launches return at once until the status
    is read, and then the workspace works again."""
    L = build_layer(D(TINY))
    d = L.dims
    layer = L.c_layer()
    ws = workspace(d, 1)
    hdr = ws[:256].view(torch.int32)
    hdr[4] = 1  # bar_extra
    h = torch.from_numpy(G.hidden_states(G.SEED, 1, 1, 256)).cuda()
    h0 = h.clone()
    M.moe_layer_decode(layer, h, ws)
    torch.cuda.synchronize()
    assert M.moe_get_device_status(ws) == 4  # MOE_ERR_TIMEOUT; header reset
    M.moe_layer_decode(layer, h0, ws)
    assert M.moe_get_device_status(ws) == 0
    ref = L.oracle(G.hidden_states(G.SEED, 1, 1, 256)[0])
    assert rel_err(h0.cpu().numpy()[0], ref["y"]) <= REL_TOL
